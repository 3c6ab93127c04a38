// General tcgen05 GEMM for the large contractions of the backward pass,
//   C[M, N] = A[M, K] B[K, N],  bf16 operands, fp32 accumulation in TMEM,
// with either operand stored either way round:
//   A_MN = false: A is a row-major [M, K] matrix (K-major); true: A is the
//                 transpose of a row-major [K, M] matrix (M-major);
//   B_KM = false: B is a row-major [K, N] matrix (N-major); true: B is the
//                 transpose of a row-major [N, K] matrix (K-major).
// Results leave through TMA from per-warp swizzled staging boxes: bf16 as
// stores; fp32 as stores, or as TMA reduce-adds when accumulating into C or
// when several CTAs split K and sum into one zeroed tile.
//
// Batched form: independent products stacked along the stored rows of each
// operand (a batch never shares a 128-row tile or a 64-deep k-block with
// the next), one tile list over all of them.
//
// Two-product form: C = A B + A2 B2 in one accumulator, the k-blocks of the
// second product (its own A majorness, B2 stored as B) following those of
// the first, so that a sum of two contractions needs no second pass over C.
//
// Elementwise epilogues (bf16 C): each epilogue warp loads the box of an
// operand E with C's coordinates by TMA into its second staging buffer (the
// next box's load issued as soon as the current one is read) and stores
// D = swish(E) * C (with C) or D = C * swish'(E) (instead of C): the gate
// of the layer and the activation's gradient, without a separate pass.
//
// One persistent CTA per SM over 128 x 256 output tiles (x split), static
// round robin.  Warp 0 streams 64-deep k-blocks of A and B into a 4-stage
// ring of 128-byte-swizzled boxes with TMA; one thread of warp 1 issues
// tcgen05.mma (M = 128, N = 256, K = 16) into one of two TMEM accumulators;
// warps 2-5 drain the other with tcgen05.ld (one TMEM lane quarter each).
#include <cuda_bf16.h>

#include "flash_gau_internal.h"
#include "sm103_ptx.cuh"
#include "tma_host.h"

namespace flashgau {
namespace {

using namespace ptx;

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;       // 16 KB
constexpr int B_BYTES = BN * BK * 2;       // 32 KB
constexpr int BOX_BYTES = 64 * 64 * 2;     // one 64 x 64 box, 8 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int ACC_COLS = 256;
constexpr int TMEM_COLS = 2 * ACC_COLS;
constexpr int NUM_THREADS = 192;
constexpr int STG_BYTES = 32 * 128;  // one 32-row x 128-byte store box
constexpr int STG_OFF = STAGES * STAGE_BYTES;  // two boxes per epilogue warp
constexpr int TILE_BYTES = STG_OFF + 4 * 2 * STG_BYTES;
constexpr int SMEM_BYTES = TILE_BYTES + 1024 /*align*/ + 256 /*barriers*/;

struct AnyParams {
  int M, N, K;
  int K2, a2_mn, b2_div;  // second product: depth, A2 majorness, B2 batch divisor
  int m_tiles, n_tiles, splits, total;
  int kb_split;  // k-blocks per split
  int atomic;    // fp32: add into C (zeroed by the caller) instead of storing
  float alpha;   // fp32 output scale
  int b_div;     // B's batch = the tile's batch / b_div
  int kbox_rows; // rows of a K-major B box: min(256, N)
  int *status;
};

struct Smem {
  uint64_t full[STAGES], empty[STAGES];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t drain;
  uint64_t ebar[4];  // per epilogue warp: its E box landed
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

struct Tile {
  int z, mt, nt, kb0, kb1;
};
__device__ __forceinline__ Tile tile_of(const AnyParams &p, int t) {
  Tile x;
  // split slowest: the CTAs of one round work on the same K range, whose
  // operand rows then stay in L2 for every output tile that reads them
  const int out_tiles = p.total / p.splits;
  const int split = t / out_tiles, rem = t % out_tiles;
  x.nt = rem % p.n_tiles;
  x.mt = (rem / p.n_tiles) % p.m_tiles;
  x.z = rem / (p.n_tiles * p.m_tiles);
  const int kblocks = (p.K + p.K2) / BK;
  x.kb0 = split * p.kb_split;
  x.kb1 = min(kblocks, x.kb0 + p.kb_split);
  return x;
}

template <bool A_MN, bool B_KM, bool OUT_BF16, int EPI = kEpiNone>
__global__ void __launch_bounds__(NUM_THREADS, 1)
tc_gemm_any_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmA2,
                   const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ CUtensorMap tmE,
                   const __grid_constant__ CUtensorMap tmD, const AnyParams p) {
  static_assert(EPI == kEpiNone || OUT_BF16, "elementwise epilogues take a bf16 C");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *tiles = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Smem *sm = reinterpret_cast<Smem *>(tiles + TILE_BYTES);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(smem_u32(&sm->full[i]), 1);
      mbar_init(smem_u32(&sm->empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sm->acc_full[i]), 1);
      mbar_init(smem_u32(&sm->acc_empty[i]), 4);  // one arrival per epilogue warp
    }
    mbar_init(smem_u32(&sm->drain), 1);
    for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&sm->ebar[i]), 1);
    sm->abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm->tmem_base), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = sm->tmem_base;
  // launched with programmatic dependent launch: the setup above overlaps
  // the previous kernel's tail; wait for it before any operand or output
  // access, and let the next kernel be scheduled
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (elect_one()) {
      int stage = 0;
      uint32_t phase = 0;
      for (int t = blockIdx.x; t < p.total && !sm->abort_flag; t += gridDim.x) {
        const Tile x = tile_of(p, t);
        const int m0 = x.mt * BM, n0 = x.nt * BN, nsz = min(BN, p.N - n0);
        // this batch's first stored row of A and of B (and of A2, B2)
        const int za = x.z * (A_MN ? p.K : p.M);
        const int zb = (x.z / p.b_div) * (B_KM ? p.N : p.K);
        const int za2 = x.z * (p.a2_mn ? p.K2 : p.M);
        const int zb2 = (x.z / p.b2_div) * (B_KM ? p.N : p.K2);
        const int kb_one = p.K / BK;  // k-blocks of the first product
        for (int kb = x.kb0; kb < x.kb1; ++kb) {
          if (!mbar_wait(smem_u32(&sm->empty[stage]), phase ^ 1, &sm->abort_flag)) {
            raise_timeout(sm, p.status);
            break;
          }
          const uint32_t full = smem_u32(&sm->full[stage]);
          uint8_t *sA = tiles + stage * STAGE_BYTES;
          uint8_t *sB = sA + A_BYTES;
          // a K-major B box is 256 rows whatever the tile's width (rows past
          // N are zero-filled and counted)
          const uint32_t b_bytes =
              B_KM ? (uint32_t)p.kbox_rows * 128u : (uint32_t)(nsz / 64) * BOX_BYTES;
          mbar_arrive_expect_tx(full, A_BYTES + b_bytes);
          // the first product's k-block, or the second's
          const bool two = kb >= kb_one;
          const int k = two ? kb - kb_one : kb;
          const CUtensorMap *ta = two ? &tmA2 : &tmA, *tb = two ? &tmB2 : &tmB;
          const bool amn = two ? p.a2_mn != 0 : A_MN;
          const int zA = two ? za2 : za, zB = two ? zb2 : zb;
          if (amn) {
            // [K, M] storage: 64 k-rows of two 64-column blocks of M
            tma_load_2d(smem_u32(sA), ta, full, m0, zA + k * BK);
            tma_load_2d(smem_u32(sA + BOX_BYTES), ta, full, m0 + 64, zA + k * BK);
          } else {
            tma_load_2d(smem_u32(sA), ta, full, k * BK, zA + m0);
          }
          if (B_KM) {
            tma_load_2d(smem_u32(sB), tb, full, k * BK, zB + n0);
          } else {
            for (int j = 0; j < nsz / 64; ++j)
              tma_load_2d(smem_u32(sB + j * BOX_BYTES), tb, full, n0 + j * 64, zB + k * BK);
          }
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    if (elect_one()) {
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      for (int t = blockIdx.x; t < p.total && !sm->abort_flag; t += gridDim.x, ++local) {
        const Tile x = tile_of(p, t);
        const int nsz = min(BN, p.N - x.nt * BN);
        const int acc = local & 1;
        if (!mbar_wait(smem_u32(&sm->acc_empty[acc]), ((local >> 1) & 1) ^ 1, &sm->abort_flag)) {
          raise_timeout(sm, p.status);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
        const int kb_one = p.K / BK;
        bool ok = true;
        for (int kb = x.kb0; kb < x.kb1; ++kb) {
          const bool amn = kb >= kb_one ? p.a2_mn != 0 : A_MN;
          const uint32_t idesc = idesc_bf16_f32(BM, nsz, amn ? 1 : 0, B_KM ? 0 : 1);
          if (!mbar_wait(smem_u32(&sm->full[stage]), phase, &sm->abort_flag)) {
            raise_timeout(sm, p.status);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = smem_u32(tiles + stage * STAGE_BYTES);
          // K-major: 16 elements (32 B) per step inside the swizzle atom;
          // MN-major: 16 k-rows of 128 B per step, 64-wide blocks 8 KB apart
          const uint64_t da = amn ? sw128_desc(sA, BOX_BYTES, 1024) : sw128_desc(sA, 16, 1024);
          const uint64_t db = B_KM ? sw128_desc(sA + A_BYTES, 16, 1024)
                                   : sw128_desc(sA + A_BYTES, BOX_BYTES, 1024);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            mma_f16_ss(d_tmem, desc_advance(da, k * (amn ? 2048 : 32)),
                       desc_advance(db, k * (B_KM ? 32 : 2048)), idesc, kb != x.kb0 || k != 0);
          mma_commit(smem_u32(&sm->empty[stage]));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit(smem_u32(&sm->acc_full[acc]));
      }
      // every MMA this thread issued has completed once `drain` flips
      mma_commit(smem_u32(&sm->drain));
      if (!mbar_wait(smem_u32(&sm->drain), 0)) raise_timeout(sm, p.status);
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    uint8_t *stg = tiles + STG_OFF + (warp - 2) * 2 * STG_BYTES;
    // elementwise epilogues: this warp's E boxes land in its second buffer
    uint8_t *ebox = stg + STG_BYTES;
    const uint32_t ebar = smem_u32(&sm->ebar[warp - 2]);
    uint32_t e_issued = 0, e_used = 0;
    auto load_e = [&](int t) {  // box 0 of tile t, or nothing past the list
      if (t >= p.total) return;
      const Tile y = tile_of(p, t);
      if (lane == 0) {
        mbar_arrive_expect_tx(ebar, STG_BYTES);
        tma_load_2d(smem_u32(ebox), &tmE, ebar, y.nt * BN, y.z * p.M + y.mt * BM + quarter * 32);
      }
      ++e_issued;
    };
    if constexpr (EPI != kEpiNone) load_e(blockIdx.x);
    int local = 0, nbox = 0;
    for (int t = blockIdx.x; t < p.total && !sm->abort_flag; t += gridDim.x, ++local) {
      const Tile x = tile_of(p, t);
      const int m0 = x.z * p.M + x.mt * BM, n0 = x.nt * BN, nsz = min(BN, p.N - n0);
      const int acc = local & 1;
      if (!mbar_wait(smem_u32(&sm->acc_full[acc]), (local >> 1) & 1, &sm->abort_flag)) {
        raise_timeout(sm, p.status);
        break;
      }
      tc_fence_after();
      const int row0 = m0 + quarter * 32;
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * ACC_COLS;
      for (int c0 = 0; c0 < nsz; c0 += 64) {
        uint32_t ra[32], rb[32];
        tmem_ld32(taddr + c0, ra);
        tmem_ld32(taddr + c0 + 32, rb);
        tmem_ld_wait();
        if (c0 + 64 >= nsz) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&sm->acc_empty[acc]));
        }
        if constexpr (OUT_BF16) {
          // this row's 64 columns as bf16
          uint4 w[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint32_t *v = q < 4 ? &ra[8 * q] : &rb[8 * (q - 4)];
            w[q].x = pack_bf16(__uint_as_float(v[0]), __uint_as_float(v[1]));
            w[q].y = pack_bf16(__uint_as_float(v[2]), __uint_as_float(v[3]));
            w[q].z = pack_bf16(__uint_as_float(v[4]), __uint_as_float(v[5]));
            w[q].w = pack_bf16(__uint_as_float(v[6]), __uint_as_float(v[7]));
          }
          if constexpr (EPI != kEpiSwishGrad) {
            // into the swizzled box, then one TMA store
            if (lane == 0) tma_store_wait_read<0>();
            __syncwarp();
#pragma unroll
            for (int q = 0; q < 8; ++q) *reinterpret_cast<uint4 *>(stg + sw128_offset(lane, q)) = w[q];
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmC, smem_u32(stg), n0 + c0, row0);
              tma_store_commit();
            }
          }
          if constexpr (EPI != kEpiNone) {
            if (!mbar_wait(ebar, e_used & 1, &sm->abort_flag)) {
              raise_timeout(sm, p.status);
              break;
            }
            ++e_used;
            // D from this row's E and C values
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const uint4 ev = *reinterpret_cast<const uint4 *>(ebox + sw128_offset(lane, q));
              const uint32_t eu[4] = {ev.x, ev.y, ev.z, ev.w};
              uint32_t cu[4] = {w[q].x, w[q].y, w[q].z, w[q].w};
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const float2 ef = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&eu[j]));
                const float2 cf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&cu[j]));
                if constexpr (EPI == kEpiGate)
                  cu[j] = pack_bf16(swish_fast(ef.x) * cf.x, swish_fast(ef.y) * cf.y);
                else
                  cu[j] = pack_bf16(cf.x * swish_grad_fast(ef.x), cf.y * swish_grad_fast(ef.y));
              }
              w[q] = make_uint4(cu[0], cu[1], cu[2], cu[3]);
            }
            // the E buffer is free: the next box's load (this tile's, or the
            // first of this warp's next tile)
            fence_proxy_async_smem();
            __syncwarp();
            if (c0 + 64 < nsz) {
              if (lane == 0) {
                mbar_arrive_expect_tx(ebar, STG_BYTES);
                tma_load_2d(smem_u32(ebox), &tmE, ebar, n0 + c0 + 64, row0);
              }
              ++e_issued;
            } else {
              load_e(t + gridDim.x);
            }
            if (lane == 0) tma_store_wait_read<0>();
            __syncwarp();
#pragma unroll
            for (int q = 0; q < 8; ++q) *reinterpret_cast<uint4 *>(stg + sw128_offset(lane, q)) = w[q];
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmD, smem_u32(stg), n0 + c0, row0);
              tma_store_commit();
            }
          }
        } else {
          // two 32-column fp32 boxes, alternating between the warp's two
          // staging buffers
#pragma unroll
          for (int h = 0; h < 2; ++h, ++nbox) {
            uint8_t *box = stg + (nbox & 1) * STG_BYTES;
            if (lane == 0) tma_store_wait_read<1>();
            __syncwarp();
            const uint32_t *v = h == 0 ? ra : rb;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              float4 w = make_float4(p.alpha * __uint_as_float(v[4 * q]),
                                     p.alpha * __uint_as_float(v[4 * q + 1]),
                                     p.alpha * __uint_as_float(v[4 * q + 2]),
                                     p.alpha * __uint_as_float(v[4 * q + 3]));
              *reinterpret_cast<float4 *>(box + sw128_offset(lane, q)) = w;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              if (p.atomic) tma_reduce_add_2d(&tmC, smem_u32(box), n0 + c0 + 32 * h, row0);
              else tma_store_2d(&tmC, smem_u32(box), n0 + c0 + 32 * h, row0);
              tma_store_commit();
            }
          }
        }
      }
    }
    // an E load still in flight (a prefetch past an early exit) lands
    // before the shared memory is given up
    if constexpr (EPI != kEpiNone)
      if (e_issued > e_used) mbar_wait(ebar, e_used & 1);
    if (lane == 0) tma_store_wait<0>();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

template <bool A_MN, bool B_KM, bool OUT_BF16, int EPI = kEpiNone>
cudaError_t launch(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC,
                   const CUtensorMap &tmA2, const CUtensorMap &tmB2, const CUtensorMap &tmE,
                   const CUtensorMap &tmD, const AnyParams &p, int num_sms, cudaStream_t stream) {
  static unsigned long long configured = 0;  // one bit per device ordinal
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  auto kernel = tc_gemm_any_kernel<A_MN, B_KM, OUT_BF16, EPI>;
  if (dev < 64 && !(configured & (1ull << dev))) {
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (err != cudaSuccess) return err;
    configured |= 1ull << dev;
  }
  const int grid = p.total < num_sms ? p.total : num_sms;
  return launch_pdl(kernel, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES, stream, tmA, tmB, tmC,
                    tmA2, tmB2, tmE, tmD, p);
}

}  // namespace

cudaError_t tc_gemm_any(const GemmAnyArgs &g, cudaStream_t stream) {
  if (g.M % BM != 0 || g.N % 64 != 0 || g.K % BK != 0 || g.M <= 0 || g.N <= 0 || g.K <= 0 ||
      g.batches <= 0 || g.b_div <= 0)
    return cudaErrorInvalidValue;
  if (g.K2 < 0 || g.K2 % BK != 0 || (g.K2 > 0 && (!g.A2 || !g.B2 || g.b2_div <= 0)))
    return cudaErrorInvalidValue;
  const long long Z = g.batches, ZB = (g.batches + g.b_div - 1) / g.b_div;
  const int kbox = g.N < BN ? g.N : BN;
  CUtensorMap tmA, tmB, tmC;
  cudaError_t err;
  // A: K-major [M, K] in 64 x 128 boxes, or M-major [K, M] in 64 x 64 boxes
  if (g.a_mn) err = make_tmap_bf16_2d(&tmA, g.A, Z * g.K, g.M, g.lda, 64, 64);
  else err = make_tmap_bf16_2d(&tmA, g.A, Z * g.M, g.K, g.lda, BM, 64);
  if (err != cudaSuccess) return err;
  // B: N-major [K, N] in 64 x 64 boxes, or K-major [N, K] in boxes of
  // min(256, N) rows
  if (g.b_km) err = make_tmap_bf16_2d(&tmB, g.B, ZB * g.N, g.K, g.ldb, kbox, 64);
  else err = make_tmap_bf16_2d(&tmB, g.B, ZB * g.K, g.N, g.ldb, 64, 64);
  if (err != cudaSuccess) return err;
  // elementwise epilogues: E and D boxes as C's (C unused by kEpiSwishGrad)
  if (g.epi != kEpiNone &&
      (!g.c_bf16 || !g.E || !g.D || (g.epi != kEpiGate && g.epi != kEpiSwishGrad) ||
       (g.epi == kEpiGate && !g.C)))
    return cudaErrorInvalidValue;
  CUtensorMap tmE, tmD;
  if (g.epi != kEpiNone) {
    if ((err = make_tmap_bf16_2d(&tmE, g.E, Z * g.M, g.N, g.lde, 32, 64)) != cudaSuccess ||
        (err = make_tmap_bf16_2d(&tmD, g.D, Z * g.M, g.N, g.ldd, 32, 64)) != cudaSuccess)
      return err;
  }
  if (g.epi == kEpiSwishGrad) tmC = tmD;
  else if (g.c_bf16) err = make_tmap_bf16_2d(&tmC, g.C, Z * g.M, g.N, g.N, 32, 64);
  else err = make_tmap_f32_2d(&tmC, g.C, Z * g.M, g.N, g.N, 32, 32);
  if (err != cudaSuccess) return err;
  if (g.epi == kEpiNone) tmE = tmD = tmC;
  // the second product's operands (unused copies of the first's when none)
  CUtensorMap tmA2 = tmA, tmB2 = tmB;
  if (g.K2 > 0) {
    const long long ZB2 = (g.batches + g.b2_div - 1) / g.b2_div;
    if (g.a2_mn) err = make_tmap_bf16_2d(&tmA2, g.A2, Z * g.K2, g.M, g.lda2, 64, 64);
    else err = make_tmap_bf16_2d(&tmA2, g.A2, Z * g.M, g.K2, g.lda2, BM, 64);
    if (err != cudaSuccess) return err;
    if (g.b_km) err = make_tmap_bf16_2d(&tmB2, g.B2, ZB2 * g.N, g.K2, g.ldb2, kbox, 64);
    else err = make_tmap_bf16_2d(&tmB2, g.B2, ZB2 * g.K2, g.N, g.ldb2, 64, 64);
    if (err != cudaSuccess) return err;
  }
  AnyParams p = {};
  p.M = g.M;
  p.N = g.N;
  p.K = g.K;
  p.K2 = g.K2;
  p.a2_mn = g.a2_mn;
  p.b2_div = g.b2_div;
  p.m_tiles = g.M / BM;
  p.n_tiles = (g.N + BN - 1) / BN;
  const int kblocks = (g.K + g.K2) / BK;
  // split K when the output tiles would leave SMs idle (fp32 atomic output
  // only), at least 8 k-blocks a split: the count with the least estimated
  // time, the persistent grid's rounds times the k-blocks of a split, plus
  // for each split an fp32 reduce-add of the whole result (measured on the
  // weight gradients: about 1.8 k-block times per MB of result)
  int splits = 1;
  const int out_tiles = (int)Z * p.m_tiles * p.n_tiles;
  if (!g.c_bf16 && g.allow_split && out_tiles < g.num_sms) {
    const double out_mb = (double)Z * g.M * g.N * sizeof(float) / 1e6;
    const int max_splits = kblocks / 8 > 1 ? kblocks / 8 : 1;
    double best = 0.0;
    for (int sp = 1; sp <= max_splits; ++sp) {
      const int kbs = (kblocks + sp - 1) / sp, n = (kblocks + kbs - 1) / kbs;
      const long long rounds = ((long long)out_tiles * n + g.num_sms - 1) / g.num_sms;
      const double cost = (double)rounds * kbs + (n > 1 ? 1.8 * n * out_mb : 0.0);
      if (sp == 1 || cost < best) {
        best = cost;
        splits = n;
      }
    }
  }
  p.kb_split = (kblocks + splits - 1) / splits;
  p.splits = (kblocks + p.kb_split - 1) / p.kb_split;
  p.total = out_tiles * p.splits;
  p.alpha = g.alpha;
  p.b_div = g.b_div;
  p.kbox_rows = kbox;
  p.atomic = p.splits > 1 || g.accumulate;
  p.status = g.status;
  if (p.atomic && !g.accumulate && !g.c_zeroed) {
    // the split partial sums add into a zeroed output
    if ((err = cudaMemsetAsync(g.C, 0, (size_t)Z * g.M * g.N * sizeof(float), stream)) !=
        cudaSuccess)
      return err;
  }
  // the epilogue forms exist for an N-major B (the backward's Vh and dV)
  if (g.epi != kEpiNone && g.b_km) return cudaErrorInvalidValue;
  if (g.epi == kEpiGate)
    return g.a_mn ? launch<true, false, true, kEpiGate>(tmA, tmB, tmC, tmA2, tmB2, tmE, tmD, p,
                                                          g.num_sms, stream)
                  : launch<false, false, true, kEpiGate>(tmA, tmB, tmC, tmA2, tmB2, tmE, tmD, p,
                                                           g.num_sms, stream);
  if (g.epi == kEpiSwishGrad)
    return g.a_mn ? launch<true, false, true, kEpiSwishGrad>(tmA, tmB, tmC, tmA2, tmB2, tmE, tmD,
                                                               p, g.num_sms, stream)
                  : launch<false, false, true, kEpiSwishGrad>(tmA, tmB, tmC, tmA2, tmB2, tmE, tmD,
                                                                p, g.num_sms, stream);
  const int key = (g.a_mn ? 4 : 0) | (g.b_km ? 2 : 0) | (g.c_bf16 ? 1 : 0);
#define ANY_LAUNCH(am, bk, cb) \
  launch<am, bk, cb>(tmA, tmB, tmC, tmA2, tmB2, tmE, tmD, p, g.num_sms, stream)
  switch (key) {
    case 0: return ANY_LAUNCH(false, false, false);
    case 1: return ANY_LAUNCH(false, false, true);
    case 2: return ANY_LAUNCH(false, true, false);
    case 3: return ANY_LAUNCH(false, true, true);
    case 4: return ANY_LAUNCH(true, false, false);
    case 5: return ANY_LAUNCH(true, false, true);
    case 6: return ANY_LAUNCH(true, true, false);
    default: return ANY_LAUNCH(true, true, true);
  }
#undef ANY_LAUNCH
}

}  // namespace flashgau
