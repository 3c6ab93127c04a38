// Chunk states of mixed chunk attention and their prefix sums, one kernel:
//   State_g  = K_lin,g^T V_g   for every chunk g of C tokens
//   Prefix_g = lin_scale * sum_{h<g} State_h   (causal; else the total once)
// or, with a chunk mask (segment ids, row normalisation), lin_scale times
// the sum (or mean) of the states of the chunk's segment that it sees
// ("Transformer Quality in Linear Time", eq. 7 and eq. 8, the summands of
// the global term and their cumulative sum), bf16 operands, fp32
// accumulation in TMEM, bf16 states; the sums run in fp32.
//
// A batched GEMM (one batch per chunk: M = s = 128, N = e, K = C) run by a
// persistent CTA per SM over 128 x 256 output tiles.  Warp 0 streams
// k-blocks (64 tokens deep) into a 4-stage 128-byte-swizzled ring with TMA:
// A = K_lin^T read M-major straight from the heads buffer, B = V rows
// N-major.  One thread of warp 1 issues tcgen05.mma into one of two TMEM
// accumulators; warps 2-5 drain the other through tcgen05.ld into swizzled
// staging and TMA stores.
//
// Once every CTA's state tiles are in memory (a grid barrier: the grid is at
// most one CTA per SM and every CTA is resident before the next kernel can
// start, so all of them arrive; the wait is bounded all the same), the same
// CTAs scan the states, which are still in L2.  A work item is a range of
// columns of one batch row for all G chunks: one bulk copy per chunk brings
// it into the (now idle) tile buffers, then each thread runs the sums for 8
// consecutive columns and writes the prefix states.
#include <cuda_bf16.h>

#include "flash_gau_internal.h"
#include "sm103_ptx.cuh"
#include "tma_host.h"

namespace flashgau {
namespace {

using namespace ptx;

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;      // 16 KB
constexpr int B_BOX_BYTES = 64 * BK * 2;  // one 64-wide N block of a k-block: 8 KB
constexpr int B_BYTES = BN * BK * 2;      // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int ACC_COLS = 256;
constexpr int TMEM_COLS = 2 * ACC_COLS;
// producer warp, MMA warp, 4 epilogue warps; 6 more warps join the scan
constexpr int NUM_THREADS = 384;
constexpr int STG_BYTES = 32 * 128;                  // one 32-row x 128-byte store box
constexpr int STG_OFF = STAGES * STAGE_BYTES;        // 2 staging boxes per epilogue warp
constexpr int TILE_BYTES = STG_OFF + 4 * 2 * STG_BYTES;
constexpr int SMEM_BYTES = TILE_BYTES + 1024 /*align*/ + 256 /*barriers*/;


struct GemmParams {
  int N, K;              // output columns, contraction depth (per batch)
  int m_tiles, n_tiles;  // per batch
  int total_tiles;       // batches * m_tiles * n_tiles
  int k_rows_per_batch;  // row offset of a batch along K in the K-indexed maps
  int s;  // rows of one chunk state
  int *status;
  int *grid_bar;  // arrivals at the grid barrier, zeroed by the projection
  // prefix scan: states [B, G, s*e] -> prefixes [B, G or 1, s*e], as
  // 16-byte groups of 8 bf16
  const uint4 *state8;
  uint4 *prefix8;
  int B, G, causal;
  long long se8;
  float lin_scale;
  const int *seg;   // [B, G] segment ids or null; a change of id starts a segment
  int average;      // divide each sum by the number of chunks in it
  int per_chunk;    // one prefix per chunk (causal or segmented)
};

struct Smem {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint64_t scan_full;  // the scan phase's bulk copies of one work item
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
// one of its two staging buffers (row = lane, swizzled), then lane 0 stores
// it.  A buffer is rewritten only after the store issued from it two boxes
// earlier has finished reading shared memory.
struct Stager {
  uint8_t *buf;  // this warp's 2 x 4 KB
  int lane;
  int count = 0;
  __device__ uint8_t *begin() {
    if (lane == 0) tma_store_wait_read<1>();
    __syncwarp();
    return buf + (count & 1) * STG_BYTES;
  }
  // row data: 8 x 16 bytes
  __device__ void put(uint8_t *b, const uint4 (&w)[8]) {
#pragma unroll
    for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4 *>(b + sw128_offset(lane, c)) = w[c];
  }
  __device__ void finish(uint8_t *b, const CUtensorMap *tm, int x, int y) {
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(tm, smem_u32(b), x, y);
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

__device__ __forceinline__ void add8(float (&run)[8], const uint4 &v) {
  const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = __bfloat1622float2(h[k]);
    run[2 * k] += f.x;
    run[2 * k + 1] += f.y;
  }
}

__device__ __forceinline__ uint4 scaled8(const float (&run)[8], float scale) {
  uint4 w;
  __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&w);
#pragma unroll
  for (int k = 0; k < 4; ++k) h[k] = __floats2bfloat162_rn(scale * run[2 * k], scale * run[2 * k + 1]);
  return w;
}

// Running sums over the chunks of each batch row, all CTAs together.  Work
// item = (batch row b, columns [r0, r0 + w) in 16-byte groups): thread 0
// copies state[b][g][r0 .. r0 + w) for every chunk g into `buf` (G bulk
// copies on one barrier), then the threads scan it column by column.  The
// states were written by other CTAs of this grid (async-proxy stores,
// ordered before the grid barrier); the caller fenced the async proxy after
// the barrier.  Returns false (status ETIMEOUT) on a timed-out wait.
__device__ bool scan_states(const GemmParams &p, uint8_t *buf, int buf_bytes, Smem *sm) {
  // columns per item: the chunks' slices fit `buf`, and about one item per CTA
  long long w = buf_bytes / (16LL * p.G);
  const long long even = ((long long)p.B * p.se8 + gridDim.x - 1) / gridDim.x;
  if (even < w) w = even;
  if (w < 1) w = 1;
  const long long per_b = (p.se8 + w - 1) / w, items = p.B * per_b;
  const uint32_t bar = smem_u32(&sm->scan_full);
  const uint4 *sbuf = reinterpret_cast<const uint4 *>(buf);
  uint32_t phase = 0;
  for (long long it = blockIdx.x; it < items; it += gridDim.x, phase ^= 1) {
    const long long b = it / per_b, r0 = (it % per_b) * w;
    const int wc = (int)min(w, p.se8 - r0);  // columns of this item
    if (threadIdx.x == 0) {
      mbar_arrive_expect_tx(bar, (uint32_t)(p.G * wc * 16));
      for (int g = 0; g < p.G; ++g)
        bulk_load(smem_u32(buf + (size_t)g * wc * 16), p.state8 + (b * p.G + g) * p.se8 + r0,
                  (uint32_t)(wc * 16), bar);
    }
    // one thread waits; every thread sees the outcome after the barrier
    if (threadIdx.x == 0 && !mbar_wait(bar, phase, &sm->abort_flag)) raise_timeout(sm, p.status);
    __syncthreads();
    if (sm->abort_flag) return false;
    uint4 *pre = p.prefix8 + (p.per_chunk ? b * p.G * p.se8 : b * p.se8) + r0;
    const int *seg = p.seg ? p.seg + b * p.G : nullptr;
    const bool plain = !seg && !p.average;  // eq. 7/8 as written: the short loop
    for (int c = threadIdx.x; plain && c < wc; c += blockDim.x) {
      float run[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int g = 0; g < p.G; ++g) {
        if (p.causal) pre[(long long)g * p.se8 + c] = scaled8(run, p.lin_scale);
        add8(run, sbuf[g * wc + c]);
      }
      if (!p.causal) pre[c] = scaled8(run, p.lin_scale);
    }
    for (int c = threadIdx.x; !plain && c < wc; c += blockDim.x) {
      float run[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      int start = 0;  // first chunk of the current segment
      // non-causal: the segment's total for each of its chunks [start, end)
      auto write_total = [&](int end) {
        const float sc = p.average ? p.lin_scale / (float)(end - start) : p.lin_scale;
        const uint4 v = scaled8(run, sc);
        for (int h = start; h < end; ++h) pre[(long long)h * p.se8 + c] = v;
      };
      for (int g = 0; g < p.G; ++g) {
        if (seg && g > 0 && __ldg(seg + g) != __ldg(seg + g - 1)) {
          if (!p.causal) write_total(g);
#pragma unroll
          for (int k = 0; k < 8; ++k) run[k] = 0.f;
          start = g;
        }
        if (p.causal) {
          const int n = g - start;  // chunks this one sees
          const float sc = p.average ? (n > 0 ? p.lin_scale / (float)n : 0.f) : p.lin_scale;
          pre[(long long)g * p.se8 + c] = scaled8(run, sc);
        }
        add8(run, sbuf[g * wc + c]);
      }
      if (!p.causal) {
        if (p.per_chunk) write_total(p.G);
        else pre[c] = scaled8(run, p.average ? p.lin_scale / (float)p.G : p.lin_scale);
      }
    }
    __syncthreads();  // the buffer is refilled by the next item
  }
  return true;
}

// A_MN: A is stored M-contiguous (K_lin^T); otherwise K-contiguous.  tmC
// is the output map (bf16 [B*G*s, e], 32-row x 64-column boxes).
template <bool A_MN>
__global__ void __launch_bounds__(NUM_THREADS, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmC, const GemmParams p) {
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
      mbar_init(smem_u32(&sm->acc_empty[i]), 128);
    }
    mbar_init(smem_u32(&sm->drain), 1);
    mbar_init(smem_u32(&sm->scan_full), 1);
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
  // setup above overlaps the previous kernel's tail; its outputs are read below
  griddep_wait();
  griddep_launch_dependents();
  const uint32_t tmem_base = sm->tmem_base;
  const int kblocks = p.K / BK;
  const int tiles_per_batch = p.m_tiles * p.n_tiles;
  // Batches (chunks) are visited last first: the projection wrote the last
  // rows most recently, so their V and K_lin are still in L2; the attention
  // kernel, which walks the chunks forward, then finds in L2 the V of the
  // first chunks, read here last.
  const int n_batches = p.total_tiles / tiles_per_batch;
  auto batch_of = [&](int t) { return n_batches - 1 - t / tiles_per_batch; };

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (elect_one()) {
      int stage = 0;
      uint32_t phase = 0;
      for (int t = blockIdx.x; t < p.total_tiles && !sm->abort_flag; t += gridDim.x) {
        const int batch = batch_of(t), rem = t % tiles_per_batch;
        const int mt = rem / p.n_tiles, nt = rem % p.n_tiles;
        const int n0 = nt * BN, nboxes = min(BN, p.N - n0) / 64;
        const int krow0 = batch * p.k_rows_per_batch;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(smem_u32(&sm->empty[stage]), phase ^ 1, &sm->abort_flag)) {
            raise_timeout(sm, p.status);
            break;
          }
          const uint32_t full = smem_u32(&sm->full[stage]);
          uint8_t *sA = tiles + stage * STAGE_BYTES;
          uint8_t *sB = sA + A_BYTES;
          mbar_arrive_expect_tx(full, A_BYTES + nboxes * B_BOX_BYTES);
          if (A_MN) {
            // two 64-wide M blocks of K_lin (columns of the head), 64 tokens deep
            tma_load_2d(smem_u32(sA), &tmA, full, 0, krow0 + kb * BK);
            tma_load_2d(smem_u32(sA + A_BYTES / 2), &tmA, full, 64, krow0 + kb * BK);
          } else {
            tma_load_2d(smem_u32(sA), &tmA, full, kb * BK, mt * BM);
          }
          // V rows of this k-block, 64-blocked: the tile's column blocks
          // are consecutive, one box of 64 * nboxes flat rows
          tma_load_2d(smem_u32(sB), &tmB, full, 0,
                      (int)rb64_row(krow0 + kb * BK, n0, p.N / 64));
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
      for (int t = blockIdx.x; t < p.total_tiles && !sm->abort_flag; t += gridDim.x, ++local) {
        const int rem = t % tiles_per_batch;
        const int nt = rem % p.n_tiles;
        const int nsz = min(BN, p.N - nt * BN);
        const int acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        if (!mbar_wait(smem_u32(&sm->acc_empty[acc]), acc_phase ^ 1, &sm->abort_flag)) {
          raise_timeout(sm, p.status);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * ACC_COLS;
        const uint32_t idesc = idesc_bf16_f32(BM, nsz, A_MN ? 1 : 0, 1);
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(smem_u32(&sm->full[stage]), phase, &sm->abort_flag)) {
            raise_timeout(sm, p.status);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sA = smem_u32(tiles + stage * STAGE_BYTES);
          // A: K-major advances 16 elements (32 B) inside the swizzle atom;
          //    M-major advances 16 rows of 128 B.  B advances 16 rows.
          const uint64_t da = A_MN ? sw128_desc(sA, A_BYTES / 2, 1024) : sw128_desc(sA, 16, 1024);
          const uint64_t db = sw128_desc(sA + A_BYTES, B_BOX_BYTES, 1024);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            mma_f16_ss(d_tmem, desc_advance(da, A_MN ? k * 2048 : k * 32), desc_advance(db, k * 2048),
                       idesc, (kb | k) != 0);
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
  } else if (warp < 6) {
    // ---------------------------------------------------------- epilogue
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    Stager st{tiles + STG_OFF + (warp - 2) * 2 * STG_BYTES, lane};
    int local = 0;
    for (int t = blockIdx.x; t < p.total_tiles && !sm->abort_flag; t += gridDim.x, ++local) {
      const int batch = batch_of(t), rem = t % tiles_per_batch;
      const int mt = rem / p.n_tiles, nt = rem % p.n_tiles;
      const int n0 = nt * BN, nsz = min(BN, p.N - n0);
      const int acc = local & 1;
      if (!mbar_wait(smem_u32(&sm->acc_full[acc]), (local >> 1) & 1, &sm->abort_flag)) {
        raise_timeout(sm, p.status);
        break;
      }
      tc_fence_after();
      const int row0 = mt * BM + quarter * 32;  // first row of this warp's box
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * ACC_COLS;
      for (int c0 = 0; c0 < nsz; c0 += 64) {
        uint32_t ra[32], rb[32];
        tmem_ld32(taddr + c0, ra);
        tmem_ld32(taddr + c0 + 32, rb);
        tmem_ld_wait();
        if (c0 + 64 >= nsz) {
          tc_fence_before();
          mbar_arrive(smem_u32(&sm->acc_empty[acc]));
        }
        uint4 w[8];
        pack64(ra, rb, [](float x, int) { return x; }, w);
        uint8_t *b = st.begin();
        st.put(b, w);
        st.finish(b, &tmC, 0, (int)rb64_row(batch * p.s + row0, n0 + c0, p.N / 64));
      }
    }
    st.drain();  // this warp's bulk stores are complete
    if (lane == 0) {
      fence_proxy_async_global();
      __threadfence();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }

  // ------------------------------------------------ grid barrier, then scan
  // Every CTA arrives, also after a timeout, so that the others are not
  // left waiting; a CTA that gave up skips the scan and reports ETIMEOUT.
  if (threadIdx.x == 0) {
    __threadfence();
    red_release_gpu_add(p.grid_bar, 1);
    const uint64_t t0 = globaltimer();
    while (ld_acquire_gpu(p.grid_bar) < (int)gridDim.x) {
      if (globaltimer() - t0 > kWaitLimitNs) {
        raise_timeout(sm, p.status);
        break;
      }
      __nanosleep(64);
    }
  }
  __syncthreads();
  // the bulk copies below (async proxy) read what the barrier made visible
  fence_proxy_async_global();
  if (!sm->abort_flag) scan_states(p, tiles, TILE_BYTES, sm);
}

template <bool A_MN>
cudaError_t launch(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC,
                   const GemmParams &p, const Problem &pr) {
  static unsigned long long configured = 0;  // one bit per device ordinal
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 64 && !(configured & (1ull << dev))) {
    err = cudaFuncSetAttribute(tc_gemm_kernel<A_MN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               SMEM_BYTES);
    if (err != cudaSuccess) return err;
    configured |= 1ull << dev;
  }
  const int grid = p.total_tiles < pr.num_sms ? p.total_tiles : pr.num_sms;
  return launch_pdl(tc_gemm_kernel<A_MN>, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES, pr.stream,
                    tmA, tmB, tmC, p);
}

GemmParams base_params(const Problem &pr) {
  GemmParams p = {};
  p.status = pr.status;
  p.grid_bar = pr.status + kGridBarrierWord;
  p.s = pr.s;
  return p;
}

}  // namespace

cudaError_t tc_chunk_state_scan_bf16(const Problem &pr) {
  // a zero global term: nothing to compute (the attention reads no prefix)
  if (pr.lin_off) return cudaSuccess;
  // batch = chunk (b*G + g): State[chunk] = K_lin[chunk rows]^T V[chunk rows]
  const __nv_bfloat16 *Kl = (const __nv_bfloat16 *)pr.heads + 3 * pr.M * pr.s;
  CUtensorMap tmA, tmB, tS;
  cudaError_t err;
  if ((err = make_tmap_bf16_2d(&tmA, Kl, pr.M, pr.s, pr.s, BK, 64)) != cudaSuccess) return err;
  // V and the states in 64 x 64 blocks (flat 128-byte rows): a k-block of V
  // for a 256-column tile is one 256-row box, a state store one 32-row box
  if (pr.e % BN != 0) return cudaErrorInvalidValue;
  if ((err = make_tmap_bf16_2d(&tmB, pr.V, pr.M * pr.e / 64, 64, 64, BN, 64)) != cudaSuccess)
    return err;
  if ((err = make_tmap_bf16_2d(&tS, pr.state, (long long)pr.B * pr.G * pr.s * pr.e / 64, 64, 64,
                               32, 64)) != cudaSuccess)
    return err;
  GemmParams p = base_params(pr);
  p.N = pr.e;
  p.K = pr.C;
  p.m_tiles = 1;  // s == 128 rows
  p.n_tiles = (pr.e + BN - 1) / BN;
  p.total_tiles = pr.B * pr.G * p.n_tiles;
  p.k_rows_per_batch = pr.C;
  p.state8 = (const uint4 *)pr.state;
  p.prefix8 = (uint4 *)pr.prefix;
  p.B = pr.B;
  p.G = pr.G;
  p.causal = pr.causal;
  p.se8 = (long long)pr.s * pr.e / 8;  // s == 128
  p.lin_scale = pr.lin_scale;
  p.seg = pr.seg_ids;
  p.average = pr.chunk_average;
  p.per_chunk = pr.per_chunk;
  return launch<true>(tmA, tmB, tS, p, pr);
}

}  // namespace flashgau
