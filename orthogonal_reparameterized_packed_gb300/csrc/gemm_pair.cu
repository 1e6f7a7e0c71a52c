// The W0 GEMMs (v = u W0^T and du = dv W0) on CTA pairs: each cluster of
// two CTAs computes 256 x 256 output tiles with tcgen05.mma.cta_group::2,
// one MMA instruction covering both CTAs' 128 rows.  Per K step each CTA
// loads its own 128 rows of A and its half (128 of the 256 N rows) of B, so
// a CTA moves 32 KiB per K step instead of the 48 KiB a one-CTA 128 x 256
// tile needs.
//
// Roles, per CTA (192 threads):
//   warp 0      TMA producer (one lane), in both CTAs: waits for its own ring
//               slot to be free, loads its A rows and B half; the bytes are
//               counted on the leader CTA's (rank 0) full barrier
//   warp 1      TMEM allocation for the pair (both CTAs); in the leader one
//               lane issues every MMA of the pair and commits the slot-free
//               and accumulator-full signals to both CTAs' barriers
//   warps 2..5  epilogue, in both CTAs: its 128 accumulator rows -> bf16 ->
//               128B-swizzled staging -> TMA tile stores; then tells the
//               leader that the accumulator is free again
// Two TMEM accumulators of 256 fp32 columns let the epilogue of one tile
// overlap the main loop of the next.  Tiles: N tile fastest, so clusters
// running at the same time share A rows (W0 stays in L2).
//
// BLOCK: the block-diagonal factor in the epilogue.  N tile j of the product
// is exactly the 256 features of superblock j, so the finished tile (v or
// du) is rounded to bf16 into a 64 KiB staging tile per CTA (stored as the
// main output when one is given), which is the A operand of a second pair
// MMA with superblock j (K = 256, streamed through the operand ring) into
// the same accumulator: y = v R_j^T (forward) or dx = du P_j (dgrad).  That
// block product is issued in the middle of the next tile's main loop, so the
// tensor pipe never waits for the staging: by the time the next-but-one tile
// needs the accumulator, the block output has long been drained.  Five ring
// stages fit next to the staging tile.
//
// Every barrier wait is bounded: on expiry the CTA records
// POETX_ERR_TIMEOUT, waits (bounded) for what it issued, and leaves through
// the same final cluster barrier as a normal exit.
#include <algorithm>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace poetx {

namespace {

constexpr int kPairThreads = 192;
constexpr int kPairBN = 256;                       // N of one pair tile
constexpr int kPairA = BM * BK * 2;                // this CTA's 128 rows, one K step
constexpr int kPairB = (kPairBN / 2) * BK * 2;     // this CTA's half of B, one K step
constexpr int kPairStage = kPairA + kPairB;        // 32 KiB
constexpr int kBlockSteps = 256 / BK;              // K steps of a block product
constexpr uint32_t kPairTmemCols = 2 * kPairBN;

template <bool BLOCK>
struct PairShape {
  static constexpr int STAGES = BLOCK ? 5 : 6;
  static constexpr int RING = STAGES * kPairStage;
  // BLOCK: the 128 x 256 bf16 tile (four 128 x 64 K-major chunks);
  // otherwise per epilogue warp 32 rows x 128 B
  static constexpr int OUT = BLOCK ? BM * kPairBN * 2 : 4 * 4096;
  static constexpr int SMEM = 1024 + RING + OUT + 256;
  static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

struct PairArgs {
  int m_pairs, n_tiles, k_steps;
  int block_at;    // BLOCK: K step of a tile's main loop before which the
                   // previous tile's block product is issued
  int store_main;  // BLOCK: also store the tile before the block product
  int* status;
};

// Unit u: N tile u % n_tiles, pair of M tiles u / n_tiles.
__device__ __forceinline__ void pair_unit(int u, const PairArgs& p, int& mp, int& nt) {
  nt = u % p.n_tiles;
  mp = u / p.n_tiles;
}

// BLOCK: this thread's accumulator row (256 fp32 columns) -> bf16 into row
// `row` of the staging tile: four 128B-swizzled K-major 128 x 64 chunks, the
// layout TMA stores from and the block MMA reads A from.
__device__ __forceinline__ void pair_stage_row(uint32_t t_base, uint8_t* stage, int row) {
#pragma unroll 1
  for (int cc = 0; cc < 4; ++cc) {
    uint32_t r0[32], r1[32];
    tmem_load_32cols(t_base + cc * 64, r0);
    tmem_load_32cols(t_base + cc * 64 + 32, r1);
    tmem_load_wait();
    uint32_t w[32];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      w[j] = pack_bf16x2(r0[2 * j], r0[2 * j + 1]);
      w[16 + j] = pack_bf16x2(r1[2 * j], r1[2 * j + 1]);
    }
    uint8_t* dst = stage + cc * (BM * 128) + row * 128;
#pragma unroll
    for (int q = 0; q < 8; ++q)
      st_shared_v4(dst + ((q ^ (row & 7)) << 4), w[4 * q], w[4 * q + 1], w[4 * q + 2],
                   w[4 * q + 3]);
  }
}

// BLOCK: one lane stores its warp's 32 staged rows (four 64-column boxes).
__device__ __forceinline__ void pair_store_rows(const CUtensorMap* map, uint8_t* stage,
                                                int quarter, int col0, int row0) {
#pragma unroll
  for (int cc = 0; cc < 4; ++cc)
    tma_store_2d(map, stage + cc * (BM * 128) + quarter * 4096, col0 + cc * 64, row0);
  bulk_commit();
}

template <bool B_MN, bool BLOCK>
__global__ void __launch_bounds__(kPairThreads, 1)
    w0_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC,
                   const __grid_constant__ CUtensorMap tmR,
                   const __grid_constant__ CUtensorMap tmY, const PairArgs p) {
  using S = PairShape<BLOCK>;
  constexpr int STAGES = S::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* ring = base;                      // stage s: A (16 KiB), then B half (16 KiB)
  uint8_t* sOut = base + S::RING;            // staging
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(base + S::RING + S::OUT);  // leader
  uint64_t* empty_bar = full_bar + STAGES;    // each CTA: its slot is free
  uint64_t* tfull_bar = empty_bar + STAGES;   // [2] each CTA: accumulator ready
  uint64_t* tempty_bar = tfull_bar + 2;       // [2] leader: accumulator drained
  uint64_t* yfull_bar = tempty_bar + 2;       // [2] BLOCK, each CTA: block product done
  uint64_t* vstaged_bar = yfull_bar + 2;      // BLOCK, leader: both staging tiles written
  uint64_t* drain_bar = vstaged_bar + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int units = p.m_pairs * p.n_tiles;
  const int first = static_cast<int>(cluster_id_x());
  const int step = static_cast<int>(cluster_count_x());

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);   // the leader's producer arrives (with both CTAs' bytes)
      mbar_init(&empty_bar[s], 1);  // the leader's MMA commit
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], 8);  // four epilogue warps of each CTA
      mbar_init(&yfull_bar[a], 1);
    }
    mbar_init(vstaged_bar, 8);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmC);
    if (BLOCK) {
      tma_prefetch_desc(&tmR);
      tma_prefetch_desc(&tmY);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kPairTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before either signals the other
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  pdl_trigger();

  // the leader's barriers as seen from either CTA
  const uint32_t full0 = map_peer(smem_u32(full_bar), 0);
  const uint32_t tempty0 = map_peer(smem_u32(tempty_bar), 0);
  const uint32_t vstaged0 = map_peer(smem_u32(vstaged_bar), 0);

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      auto next_slot = [&]() -> bool {
        if (!mbar_wait_cluster(&empty_bar[stage], phase ^ 1, abort_flag)) {
          record_timeout(p.status, abort_flag);
          return false;
        }
        return true;
      };
      auto advance = [&]() {
        ++issued;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      };
      // BLOCK: superblock j, one 64-row K slice per ring slot (B half only)
      auto load_block = [&](int j) -> bool {
        for (int kc = 0; kc < kBlockSteps; ++kc) {
          if (!next_slot()) return false;
          if (leader) mbar_arrive_expect_tx(&full_bar[stage], 2 * kPairB);
          uint8_t* b_dst = ring + stage * kPairStage + kPairA;
          const uint32_t bar = full0 + static_cast<uint32_t>(stage * 8);
          const int half = static_cast<int>(rank) * (kPairBN / 2);
          if (!B_MN) {  // B[n][kk] = R_j[n][kk]: rows j*256 + n of the superblocks
            tma_load_2d_pair(b_dst, &tmR, bar, kc * BK, j * 256 + half);
          } else {  // B[n][kk] = P_j[kk][n]: rows j*256 + kk, columns n
            tma_load_2d_pair(b_dst, &tmR, bar, half, j * 256 + kc * BK);
            tma_load_2d_pair(b_dst + 8192, &tmR, bar, half + 64, j * 256 + kc * BK);
          }
          advance();
        }
        return true;
      };
      int i = 0, prev_nt = -1;
      for (int u = first; u < units && ok; u += step, ++i) {
        int mp, nt;
        pair_unit(u, p, mp, nt);
        const int a_row = mp * 2 * BM + static_cast<int>(rank) * BM;
        const int b_n = nt * kPairBN + static_cast<int>(rank) * (kPairBN / 2);
        for (int ks = 0; ks < p.k_steps; ++ks) {
          if (BLOCK && i > 0 && ks == p.block_at && !load_block(prev_nt)) {
            ok = false;
            break;
          }
          if (!next_slot()) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(&full_bar[stage], 2 * kPairStage);
          uint8_t* a_dst = ring + stage * kPairStage;
          uint8_t* b_dst = a_dst + kPairA;
          const uint32_t bar = full0 + static_cast<uint32_t>(stage * 8);
          tma_load_2d_pair(a_dst, &tmA, bar, ks * BK, a_row);
          if (!B_MN) {
            tma_load_2d_pair(b_dst, &tmB, bar, ks * BK, b_n);
          } else {
            tma_load_2d_pair(b_dst, &tmB, bar, b_n, ks * BK);
            tma_load_2d_pair(b_dst + 8192, &tmB, bar, b_n + 64, ks * BK);
          }
          advance();
        }
        prev_nt = nt;
      }
      if (BLOCK && ok && i > 0 && !load_block(prev_nt)) ok = false;
      // Before leaving: every slot this CTA filled is released again, so no
      // MMA still reads this CTA's ring and no commit is still on its way to
      // its barriers (bounded).
      const int outstanding = issued < STAGES ? static_cast<int>(issued) : STAGES;
      int st = stage;
      uint32_t ph = phase;
      for (int n = 0; n < outstanding; ++n) {
        if (--st < 0) {
          st = STAGES - 1;
          ph ^= 1;
        }
        const unsigned long long t0 = global_timer_ns();
        while (!mbar_try_wait_cluster(&empty_bar[st], ph) &&
               global_timer_ns() - t0 < (ok ? kWaitLimitNs : 10000000ull)) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // -------------------------------------------------- MMA issuer (pair)
      constexpr uint32_t IDESC = instr_desc_bf16(2 * BM, kPairBN, false, B_MN);
      const uint32_t empty_own = smem_u32(empty_bar);
      const uint32_t empty_peer = map_peer(empty_own, 1);
      const uint32_t tfull_own = smem_u32(tfull_bar);
      const uint32_t tfull_peer = map_peer(tfull_own, 1);
      const uint32_t yfull_own = smem_u32(yfull_bar);
      const uint32_t yfull_peer = map_peer(yfull_own, 1);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      uint32_t vphase = 0;
      bool ok = true;
      bool any_mma = false;
      auto wait_full = [&]() -> bool {
        if (!mbar_wait_cluster(&full_bar[stage], phase, abort_flag)) {
          record_timeout(p.status, abort_flag);
          return false;
        }
        tc_fence_after();
        return true;
      };
      auto release = [&]() {  // the slot is free in both CTAs once the MMAs have read it
        umma_commit_pair(empty_own + static_cast<uint32_t>(stage * 8));
        umma_commit_pair(empty_peer + static_cast<uint32_t>(stage * 8));
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1;
        }
      };
      // BLOCK: the staged tile of accumulator a times its superblock, into a
      auto block_mma = [&](int a) -> bool {
        if (!mbar_wait_cluster(vstaged_bar, vphase, abort_flag)) {
          record_timeout(p.status, abort_flag);
          return false;
        }
        vphase ^= 1;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(a * kPairBN);
        const uint32_t v_base = smem_u32(sOut);
        for (int kc = 0; kc < kBlockSteps; ++kc) {
          if (!wait_full()) return false;
          const uint32_t b_base = smem_u32(ring + stage * kPairStage + kPairA);
#pragma unroll
          for (int j = 0; j < BK / 16; ++j) {
            const uint64_t adesc = smem_desc_sw128(v_base + kc * (BM * 128) + j * 32, 16, 1024);
            const uint64_t bdesc = B_MN ? smem_desc_sw128(b_base + j * 2048, 8192, 1024)
                                        : smem_desc_sw128(b_base + j * 32, 16, 1024);
            umma_bf16_pair(d_tmem, adesc, bdesc, IDESC, (kc > 0 || j > 0) ? 1u : 0u);
          }
          release();
        }
        umma_commit_pair(yfull_own + static_cast<uint32_t>(a * 8));
        umma_commit_pair(yfull_peer + static_cast<uint32_t>(a * 8));
        return true;
      };
      int i = 0;
      for (int u = first; u < units && ok; u += step, ++i) {
        if (!mbar_wait_cluster(&tempty_bar[acc], acc_phase ^ 1, abort_flag)) {
          record_timeout(p.status, abort_flag);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kPairBN);
        for (int ks = 0; ks < p.k_steps; ++ks) {
          if (BLOCK && i > 0 && ks == p.block_at) {
            // the previous tile's block product, into the other accumulator
            any_mma = true;
            if (!block_mma(acc ^ 1)) {
              ok = false;
              break;
            }
          }
          if (!wait_full()) {
            ok = false;
            break;
          }
          const uint32_t a_base = smem_u32(ring + stage * kPairStage);
          const uint32_t b_base = a_base + kPairA;
#pragma unroll
          for (int j = 0; j < BK / 16; ++j) {
            const uint64_t adesc = smem_desc_sw128(a_base + j * 32, 16, 1024);
            const uint64_t bdesc = B_MN ? smem_desc_sw128(b_base + j * 2048, 8192, 1024)
                                        : smem_desc_sw128(b_base + j * 32, 16, 1024);
            umma_bf16_pair(d_tmem, adesc, bdesc, IDESC, (ks > 0 || j > 0) ? 1u : 0u);
          }
          any_mma = true;
          release();
        }
        if (!ok) break;
        umma_commit_pair(tfull_own + static_cast<uint32_t>(acc * 8));
        umma_commit_pair(tfull_peer + static_cast<uint32_t>(acc * 8));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      if (BLOCK && ok && i > 0 && !block_mma(acc ^ 1)) ok = false;
      if (!ok && any_mma) {
        // the MMAs in flight finish before TMEM is released
        umma_commit_pair(smem_u32(drain_bar));
        const unsigned long long t0 = global_timer_ns();
        while (!mbar_try_wait(drain_bar, 0) && global_timer_ns() - t0 < 10000000ull) {
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // the TMEM lanes this warp may read
    const int row = quarter * 32 + lane;  // this thread's accumulator row
    uint8_t* stg = sOut + quarter * 4096;
    uint8_t* my_row = stg + lane * 128;
    bool stores_pending = false;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = first; u < units; u += step) {
      int mp, nt;
      pair_unit(u, p, mp, nt);
      const bool got = mbar_wait_cluster(&tfull_bar[acc], acc_phase, abort_flag);
      if (!__all_sync(0xffffffffu, got)) {
        record_timeout(p.status, abort_flag);
        break;
      }
      tc_fence_after();
      const uint32_t t_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                              static_cast<uint32_t>(acc * kPairBN);
      const int out_row = mp * 2 * BM + static_cast<int>(rank) * BM + quarter * 32;
      const int out_col0 = nt * kPairBN;
      if (BLOCK) {
        // (1) the tile to bf16: the block product's A operand (and the main output)
        if (lane == 0 && stores_pending) bulk_wait_read_all();  // staging free again
        __syncwarp();
        pair_stage_row(t_base, sOut, row);
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0 && p.store_main) {
          pair_store_rows(&tmC, sOut, quarter, out_col0, out_row);
          stores_pending = true;
        }
        // the block MMA overwrites this accumulator: its reads come first
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(vstaged0);
        // (2) the block product: to bf16 and out; then the accumulator is free
        const bool ygot = mbar_wait_cluster(&yfull_bar[acc], acc_phase, abort_flag);
        if (!__all_sync(0xffffffffu, ygot)) {
          record_timeout(p.status, abort_flag);
          break;
        }
        tc_fence_after();
        if (lane == 0 && stores_pending) bulk_wait_read_all();
        __syncwarp();
        pair_stage_row(t_base, sOut, row);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(tempty0 + static_cast<uint32_t>(acc * 8));
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) {
          pair_store_rows(&tmY, sOut, quarter, out_col0, out_row);
          stores_pending = true;
        }
      } else {
#pragma unroll 1
        for (int c0 = 0; c0 < kPairBN; c0 += 64) {
          uint32_t r0[32], r1[32];
          tmem_load_32cols(t_base + c0, r0);
          tmem_load_32cols(t_base + c0 + 32, r1);
          tmem_load_wait();
          uint32_t w[32];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            w[j] = pack_bf16x2(r0[2 * j], r0[2 * j + 1]);
            w[16 + j] = pack_bf16x2(r1[2 * j], r1[2 * j + 1]);
          }
          if (lane == 0 && stores_pending) bulk_wait_read_all();  // staging free again
          __syncwarp();
#pragma unroll
          for (int q = 0; q < 8; ++q)  // 16-byte chunk q of the row, 128B-swizzled
            st_shared_v4(my_row + ((q ^ (lane & 7)) << 4), w[4 * q], w[4 * q + 1],
                         w[4 * q + 2], w[4 * q + 3]);
          fence_proxy_async_shared();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmC, stg, out_col0 + c0, out_row);
            bulk_commit();
            stores_pending = true;
          }
        }
        tc_fence_before();
        __syncwarp();
        // the accumulator is free again once both CTAs' four warps have read it
        if (lane == 0) mbar_arrive_remote(tempty0 + static_cast<uint32_t>(acc * 8));
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    if (lane == 0 && stores_pending) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still signal or read it
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kPairTmemCols);
  }
}

template <bool B_MN, bool BLOCK>
cudaError_t launch_pair(const TcGemm& g, cudaStream_t stream) {
  using S = PairShape<BLOCK>;
  auto* kernel = w0_pair_kernel<B_MN, BLOCK>;
  static bool attr_set[64] = {false};
  static int max_clusters[64] = {0};
  static std::mutex mu;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::unique_lock<std::mutex> lock(mu);
  if (!attr_set[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * sm_count());
    cfg.blockDim = dim3(kPairThreads);
    cfg.dynamicSmemBytes = S::SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorLaunchOutOfResources;
    max_clusters[dev] = n;
    attr_set[dev] = true;
  }
  const int cmax = max_clusters[dev];
  lock.unlock();

  CUtensorMap tmA, tmB, tmC, tmR, tmY;
  if (!make_map(&tmA, g.A.ptr, g.A.rows, g.A.cols, g.A.pitch, 2, 64, BM))
    return cudaErrorInvalidValue;
  if (!make_map(&tmB, g.B.ptr, g.B.rows, g.B.cols, g.B.pitch, 2, 64,
                B_MN ? 64 : kPairBN / 2))
    return cudaErrorInvalidValue;
  const bool main_out = g.epi.out_bf16 != nullptr;
  if (main_out && !make_map(&tmC, g.epi.out_bf16, g.epi.out_rows, g.epi.ld, g.epi.ld, 2, 64, 32))
    return cudaErrorInvalidValue;
  if (BLOCK) {
    if (!make_map(&tmR, g.blk.ptr, g.blk.rows, g.blk.cols, g.blk.pitch, 2, 64,
                  B_MN ? 64 : kPairBN / 2))
      return cudaErrorInvalidValue;
    if (!make_map(&tmY, g.out_blk, g.epi.out_rows, g.epi.ld, g.epi.ld, 2, 64, 32))
      return cudaErrorInvalidValue;
    if (!main_out) tmC = tmY;  // never stored through
  } else {
    tmR = tmA;  // unused
    tmY = tmA;
  }
  PairArgs p;
  p.m_pairs = (g.M + 2 * BM - 1) / (2 * BM);
  p.n_tiles = g.N / kPairBN;
  p.k_steps = (g.K + BK - 1) / BK;
  p.block_at = std::min(32, p.k_steps / 2);
  p.store_main = main_out ? 1 : 0;
  p.status = device_status_ptr();
  const long long units = static_cast<long long>(p.m_pairs) * p.n_tiles;
  if (units <= 0) return cudaSuccess;
  const int clusters = static_cast<int>(std::min<long long>(units, cmax));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters);
  cfg.blockDim = dim3(kPairThreads);
  cfg.dynamicSmemBytes = S::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  prof_begin(g.tag, stream);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, tmA, tmB, tmC, tmR, tmY, p);
  prof_end(g.tag, stream);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t w0_pair_run(const TcGemm& g, cudaStream_t stream) {
  if (g.M <= 0 || g.N <= 0 || g.K <= 0) return cudaSuccess;
  if (g.batches != 1 || g.splits != 1 || g.N % kPairBN != 0 || g.K % 256 != 0 ||
      g.A.mn_major || g.epi.out_f32 != nullptr || g.epi.out_rows <= 0)
    return cudaErrorInvalidValue;
  if (g.out_blk != nullptr) {  // block factor in the epilogue (same major-ness as B)
    if (g.blk.mn_major != g.B.mn_major) return cudaErrorInvalidValue;
    if (!g.B.mn_major) return launch_pair<false, true>(g, stream);
    return launch_pair<true, true>(g, stream);
  }
  if (g.epi.out_bf16 == nullptr) return cudaErrorInvalidValue;
  if (!g.B.mn_major) return launch_pair<false, false>(g, stream);
  return launch_pair<true, false>(g, stream);
}

}  // namespace poetx
