// Tensor-core contraction engine for sm_103a: C = A * B^T per batch, bf16
// operands staged by TMA into 128-byte-swizzled shared memory, tcgen05.mma
// accumulating in TMEM, epilogue straight from TMEM.
//
// One persistent CTA per SM, warp-specialised:
//   warp 0      TMA producer (one elected lane)
//   warp 1      TMEM allocator + MMA issuer (one elected lane)
//   warps 2..5  epilogue: TMEM -> registers -> global
// Two TMEM accumulators (2 x BN fp32 columns) let the epilogue of tile i
// overlap the main loop of tile i+1.
//
// Variants (template parameters):
//   B_RES  the B operand of one (batch, N tile) stays resident in shared
//          memory while the CTA walks a contiguous run of M tiles; only A
//          streams through the ring.  Used by the block-diagonal transforms,
//          whose B is one b x b block reused by every token tile.
//   EPI    EPI_ROWS: each thread owns one accumulator row and applies the
//          general EpiArgs (scale, fp32 addends, diagonal shift, fp32/bf16
//          outputs) with 16-byte stores.  EPI_TMA_BF16 / EPI_TMA_F32: plain
//          stores of one output; each warp writes its 32-row chunk into a
//          128B-swizzled staging buffer and one lane issues a TMA tile store.
//          EPI_BLOCK: the block-diagonal factor applied in the epilogue.  The
//          output tile (128 rows x 256 = one 256 x 256 block's columns) is
//          rounded to bf16 into a 64 KiB staging tile (stored as the main
//          output when one is given), which then is the A operand of a second
//          MMA with that block (streamed through the ring) into the same
//          accumulator; the result is the block output.  Three ring stages
//          leave room for the staging tile.
//   CL2    clusters of two CTAs computing adjacent M tiles of one N tile
//          (each loads its own operands).
//          When the last round of tiles would leave clusters idle, its tiles
//          are spread one per cluster instead, the two CTAs taking the two
//          halves of the K steps; each CTA sends the partial sums of the
//          rows its peer finishes into the peer's (then idle) ring through
//          distributed shared memory and adds the peer's for its own rows.
//
// Every barrier wait is bounded: on expiry the CTA records
// POETX_ERR_TIMEOUT, drains what it issued, frees TMEM and returns.
#include <algorithm>
#include <cstdio>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace poetx {

namespace {

constexpr int NUM_THREADS = 192;
constexpr int kResBytes = 128 * 1024;

enum { EPI_ROWS = 0, EPI_TMA_BF16 = 1, EPI_TMA_F32 = 2, EPI_BLOCK = 3 };

template <int BN, bool B_RES, int EPI>
struct TcShape {
  // resident B: only A streams, and a fifth 16 KiB stage still fits
  static constexpr int STAGES = EPI == EPI_BLOCK ? 3 : (B_RES ? 5 : 4);
  static constexpr int A_BYTES = BM * BK * 2;  // 16 KB
  static constexpr int B_BYTES = BN * BK * 2;  // one K step of B: 16 or 32 KB
  static constexpr int RING = B_RES ? STAGES * A_BYTES : STAGES * (A_BYTES + B_BYTES);
  static constexpr int RES = B_RES ? kResBytes : 0;
  static constexpr int MAX_RES_KSTEPS = kResBytes / B_BYTES;
  // TMA-store staging: per warp 32 rows x 128 B; EPI_BLOCK: the 128 x 256 bf16 tile
  static constexpr int OUT_STAGE = EPI == EPI_ROWS ? 0 : (EPI == EPI_BLOCK ? BM * BN * 2 : 4 * 4096);
  static constexpr int SMEM = 1024 + RING + RES + OUT_STAGE + 256;
  static constexpr uint32_t TMEM_COLS = 2 * BN;
  static_assert(EPI != EPI_BLOCK || (BN == 256 && !B_RES), "block epilogue: 256-wide tiles");
  static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

constexpr int kBlockKSteps = 256 / BK;  // K steps of the epilogue's 256 x 256 block

struct TcKernelArgs {
  int m_tiles, n_tiles, splits, batches;
  int m_pairs;  // CL2: pairs of M tiles, one per cluster of two CTAs
  // CL2 work items: units [0, tail_first) whole; each later unit becomes two
  // items (its two M tiles), each taken by one cluster whose CTAs split its
  // K steps in halves of k_half; items = tail_first + 2 * (units - tail_first)
  int tail_first, items, k_half;
  int k_steps_total, k_steps_per_split;
  int a_mn_per_g, a_k_per_g, b_mn_per_g, b_k_per_g;
  EpiArgs epi;
  int store_main;  // EPI_BLOCK: also store the tile before the block (tmC)
  int* status;
};

// Tile order: non-resident variants walk N fastest (consecutive tiles of a
// CTA's wave share the A rows); resident-B variants walk M fastest so a CTA's
// contiguous run of tiles keeps one B.
template <bool B_RES>
__device__ __forceinline__ void decode_tile(int t, const TcKernelArgs& p, int& g, int& sp, int& mt,
                                            int& nt) {
  if (B_RES) {
    mt = t % p.m_tiles;
    t /= p.m_tiles;
    nt = t % p.n_tiles;
    t /= p.n_tiles;
  } else {
    nt = t % p.n_tiles;
    t /= p.n_tiles;
    mt = t % p.m_tiles;
    t /= p.m_tiles;
  }
  sp = t % p.splits;
  g = t / p.splits;
}

// CL2: a cluster of two CTAs takes work units (g, split, M pair, N tile); CTA
// rank r of the cluster computes M tile 2 * pair + r, so the two share B.
template <bool B_RES, bool CL2>
__device__ __forceinline__ void decode_unit(int t, const TcKernelArgs& p, uint32_t crank, int& g,
                                            int& sp, int& mt, int& nt) {
  if (CL2) {
    nt = t % p.n_tiles;
    t /= p.n_tiles;
    mt = 2 * (t % p.m_pairs) + static_cast<int>(crank);
    t /= p.m_pairs;
    sp = t % p.splits;
    g = t / p.splits;
  } else {
    decode_tile<B_RES>(t, p, g, sp, mt, nt);
  }
}

// One CTA's share of a work item: tile (g, sp, mt, nt) over K steps
// [ks0, ks1).  split: a CL2 tail item, whose two CTAs accumulate the two K
// halves of the same tile and combine them in the epilogue.
struct WorkItem {
  int g, sp, mt, nt, ks0, ks1;
  bool split;
};

template <bool B_RES, bool CL2>
__device__ __forceinline__ WorkItem decode_item(int t, const TcKernelArgs& p, uint32_t crank) {
  WorkItem w;
  w.split = CL2 && t >= p.tail_first;
  if (w.split) {
    // item i of the tail: M tile (i & 1) of unit tail_first + i / 2
    const int i = t - p.tail_first;
    decode_unit<B_RES, CL2>(p.tail_first + i / 2, p, static_cast<uint32_t>(i & 1), w.g, w.sp,
                            w.mt, w.nt);
    w.ks0 = w.sp * p.k_steps_per_split + static_cast<int>(crank) * p.k_half;
    w.ks1 = min(w.ks0 + p.k_half, p.k_steps_total);
  } else {
    decode_unit<B_RES, CL2>(t, p, crank, w.g, w.sp, w.mt, w.nt);
    w.ks0 = w.sp * p.k_steps_per_split;
    w.ks1 = min(w.ks0 + p.k_steps_per_split, p.k_steps_total);
  }
  return w;
}

// Tiles of this CTA: resident variants take a contiguous run, others stride
// (CL2: over clusters).
template <bool B_RES, bool CL2>
struct TileRange {
  int first, end, step;
  __device__ explicit TileRange(int num_tiles) {
    if (CL2) {
      first = static_cast<int>(cluster_id_x());
      end = num_tiles;
      step = static_cast<int>(cluster_count_x());
    } else if (B_RES) {
      const int per = (num_tiles + gridDim.x - 1) / gridDim.x;
      first = blockIdx.x * per;
      end = min(first + per, num_tiles);
      step = 1;
    } else {
      first = blockIdx.x;
      end = num_tiles;
      step = gridDim.x;
    }
  }
};

// Split items: a 64-row half tile of fp32 partial sums in the peer's ring,
// 1 KiB per row (lr); the 16-byte chunk q of a row sits at chunk q ^ (lr & 7)
// of its 128-byte group, so eight consecutive rows hit distinct banks.
__device__ __forceinline__ uint32_t xchg_offset(int q, int lr) {
  return static_cast<uint32_t>(lr * 1024 + (((q & ~7) | ((q ^ lr) & 7)) << 4));
}

__device__ __forceinline__ void add_f4(uint32_t* r, const float4 v) {
  r[0] = __float_as_uint(__uint_as_float(r[0]) + v.x);
  r[1] = __float_as_uint(__uint_as_float(r[1]) + v.y);
  r[2] = __float_as_uint(__uint_as_float(r[2]) + v.z);
  r[3] = __float_as_uint(__uint_as_float(r[3]) + v.w);
}

// EPI_BLOCK: this warp's 32 accumulator rows (256 fp32 columns) -> bf16 rows
// of the 128 x 256 staging tile, laid out as four 128B-swizzled K-major
// 128 x 64 chunks (the form TMA stores from and the MMA reads A from).
__device__ __forceinline__ void stage_rows_bf16(uint32_t t_base, uint8_t* stage, int row) {
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
      st_shared_v4(dst + ((q ^ (row & 7)) << 4), w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
  }
}

// One lane stores this warp's 32 staged rows (four 64-column boxes).
__device__ __forceinline__ void store_staged_rows(const CUtensorMap* map, uint8_t* stage,
                                                  int quarter, int col0, int row0) {
#pragma unroll
  for (int cc = 0; cc < 4; ++cc)
    tma_store_2d(map, stage + cc * (BM * 128) + quarter * 4096, col0 + cc * 64, row0);
  bulk_commit();
}

template <bool A_MN, bool B_MN, int BN, bool B_RES, int EPI, bool CL2>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC,
                   const __grid_constant__ CUtensorMap tmR,
                   const __grid_constant__ CUtensorMap tmY, const TcKernelArgs p) {
  using S = TcShape<BN, B_RES, EPI>;
  static_assert(!CL2 || (EPI == EPI_TMA_BF16 && !B_RES && BN == 256), "clusters: W0 GEMMs");
  static_assert(!CL2 || S::STAGES * S::A_BYTES >= 64 * BN * 4, "split items: 64 fp32 rows in sA");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  constexpr int STAGES = S::STAGES;
  uint8_t* sA = base;                        // STAGES x A tile
  uint8_t* sB = base + STAGES * S::A_BYTES;  // STAGES x B tile (streamed variants)
  uint8_t* sRes = base + S::RING;            // resident B (B_RES)
  uint8_t* sOut = base + S::RING + S::RES;   // TMA-store staging (EPI_TMA_*)
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(base + S::RING + S::RES + S::OUT_STAGE);
  uint64_t* empty_bar = full_bar + STAGES;
  uint64_t* tfull_bar = empty_bar + STAGES;  // [2]
  uint64_t* tempty_bar = tfull_bar + 2;      // [2]
  uint64_t* drain_bar = tempty_bar + 2;
  uint64_t* bfull_bar = drain_bar + 1;
  uint64_t* bempty_bar = bfull_bar + 1;
  uint64_t* vstaged_bar = bempty_bar + 1;  // EPI_BLOCK: staging tile written (4 warps)
  uint64_t* yfull_bar = vstaged_bar + 1;   // EPI_BLOCK: block MMA done
  uint64_t* xready_bar = yfull_bar + 1;    // CL2 split item: the peer's ring is free
  uint64_t* xfull_bar = xready_bar + 1;    // CL2 split item: the peer's partial rows are here
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xfull_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t crank = CL2 ? cluster_ctarank() : 0u;
  const int num_tiles = CL2 ? p.items : p.batches * p.splits * p.m_tiles * p.n_tiles;
  const TileRange<B_RES, CL2> range(num_tiles);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], 4);
    }
    mbar_init(drain_bar, 1);
    mbar_init(bfull_bar, 1);
    mbar_init(bempty_bar, 1);
    mbar_init(vstaged_bar, 4);
    mbar_init(yfull_bar, 1);
    mbar_init(xready_bar, 1);
    mbar_init(xfull_bar, 64);  // the peer's two sending warps, every lane
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (EPI != EPI_ROWS) tma_prefetch_desc(&tmC);
    if (EPI == EPI_BLOCK) {
      tma_prefetch_desc(&tmR);
      tma_prefetch_desc(&tmY);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, S::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  if (CL2) cluster_sync();  // the peer's barriers exist before the peer signals them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();  // the predecessor's outputs are complete from here on
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      int res_key = -1, res_loads = 0;
      int prev_nt = -1;
      // EPI_BLOCK: the 256 x 256 block of N tile j, one K step per ring stage (B slot)
      auto load_block = [&](int j) -> bool {
        for (int kc = 0; kc < kBlockKSteps; ++kc) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1, abort_flag)) {
            record_timeout(p.status, abort_flag);
            return false;
          }
          mbar_arrive_expect_tx(&full_bar[stage], S::B_BYTES);
          uint8_t* b_dst = sB + stage * S::B_BYTES;
          const int blk_row = j * BN;  // block j covers output columns j*256 ..
          if (!B_MN) {
            tma_load_2d(b_dst, &tmR, &full_bar[stage], kc * BK, blk_row);
          } else {
#pragma unroll
            for (int c = 0; c < BN / 64; ++c)
              tma_load_2d(b_dst + c * 8192, &tmR, &full_bar[stage], 64 * c, blk_row + kc * BK);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        return true;
      };
      for (int tile = range.first; tile < range.end && ok; tile += range.step) {
        const WorkItem item = decode_item<B_RES, CL2>(tile, p, crank);
        const int g = item.g, mt = item.mt, nt = item.nt, ks0 = item.ks0, ks1 = item.ks1;
        const int a_mn = g * p.a_mn_per_g + mt * BM;
        const int b_mn = g * p.b_mn_per_g + nt * BN;
        if (B_RES) {
          const int key = g * p.n_tiles + nt;
          if (key != res_key) {
            // the previous resident B is free once the MMAs that read it are done
            if (!mbar_wait(bempty_bar, (res_loads & 1) ^ 1, abort_flag)) {
              record_timeout(p.status, abort_flag);
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(bfull_bar, p.k_steps_total * S::B_BYTES);
            for (int kc = 0; kc < p.k_steps_total; ++kc) {
              const int b_k = g * p.b_k_per_g + kc * BK;
              uint8_t* dst = sRes + kc * S::B_BYTES;
              if (!B_MN) {
                tma_load_2d(dst, &tmB, bfull_bar, b_k, b_mn);
              } else {
#pragma unroll
                for (int c = 0; c < BN / 64; ++c)
                  tma_load_2d(dst + c * 8192, &tmB, bfull_bar, b_mn + 64 * c, b_k);
              }
            }
            res_key = key;
            ++res_loads;
          }
        }
        for (int ks = ks0; ks < ks1; ++ks) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1, abort_flag)) {
            record_timeout(p.status, abort_flag);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full_bar[stage], S::A_BYTES + (B_RES ? 0 : S::B_BYTES));
          const int a_k = g * p.a_k_per_g + ks * BK;
          uint8_t* a_dst = sA + stage * S::A_BYTES;
          if (!A_MN) {
            tma_load_2d(a_dst, &tmA, &full_bar[stage], a_k, a_mn);
          } else {
            tma_load_2d(a_dst, &tmA, &full_bar[stage], a_mn, a_k);
            tma_load_2d(a_dst + 8192, &tmA, &full_bar[stage], a_mn + 64, a_k);
          }
          if (!B_RES && CL2) {
            // each CTA of the cluster loads its whole B tile itself (split
            // items read different K steps; whole items the same tile, which
            // L2 serves twice)
            const int b_k = g * p.b_k_per_g + ks * BK;
            uint8_t* b_dst = sB + stage * S::B_BYTES;
            if (!B_MN) {
#pragma unroll
              for (int hh = 0; hh < 2; ++hh)
                tma_load_2d(b_dst + hh * (BN / 2) * 128, &tmB, &full_bar[stage], b_k,
                            b_mn + hh * (BN / 2));
            } else {
#pragma unroll
              for (int c = 0; c < BN / 64; ++c)
                tma_load_2d(b_dst + c * 8192, &tmB, &full_bar[stage], b_mn + 64 * c, b_k);
            }
          } else if (!B_RES) {
            const int b_k = g * p.b_k_per_g + ks * BK;
            uint8_t* b_dst = sB + stage * S::B_BYTES;
            if (!B_MN) {
              tma_load_2d(b_dst, &tmB, &full_bar[stage], b_k, b_mn);
            } else {
#pragma unroll
              for (int c = 0; c < BN / 64; ++c)
                tma_load_2d(b_dst + c * 8192, &tmB, &full_bar[stage], b_mn + 64 * c, b_k);
            }
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (EPI == EPI_BLOCK && ok) {
          // the previous tile's block goes after this tile's main loop: its
          // MMA then waits for nothing the epilogue is still doing
          if (prev_nt >= 0 && !load_block(prev_nt)) {
            ok = false;
            break;
          }
          prev_nt = nt;
        }
      }
      if (EPI == EPI_BLOCK && ok && prev_nt >= 0 && !load_block(prev_nt)) ok = false;
      if (!ok) {
        // Let the copies already issued land before the CTA exits.
        const int outstanding = issued < STAGES ? static_cast<int>(issued) : STAGES;
        int st = stage;
        uint32_t ph = phase;
        for (int i = 0; i < outstanding; ++i) {
          if (--st < 0) {
            st = STAGES - 1;
            ph ^= 1;
          }
          const unsigned long long t0 = global_timer_ns();
          while (!mbar_try_wait(&full_bar[st], ph) && global_timer_ns() - t0 < 10000000ull) {
          }
        }
        if (B_RES && res_loads > 0) {
          const unsigned long long t0 = global_timer_ns();
          while (!mbar_try_wait(bfull_bar, (res_loads - 1) & 1) &&
                 global_timer_ns() - t0 < 10000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------- MMA issuer
      constexpr uint32_t IDESC = instr_desc_bf16(BM, BN, A_MN, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      bool any_mma = false;
      int res_key = -1, res_loads = 0;
      uint32_t vphase = 0;
      bool have_prev = false;
      // EPI_BLOCK: once the epilogue has staged a tile in bf16, multiply it by
      // its block (from the ring) into accumulator d, then signal yfull
      auto block_mma = [&](uint32_t d) -> bool {
        if (!mbar_wait(vstaged_bar, vphase, abort_flag)) {
          record_timeout(p.status, abort_flag);
          return false;
        }
        vphase ^= 1;
        tc_fence_after();
        const uint32_t v_base = smem_u32(sOut);
        for (int kc = 0; kc < kBlockKSteps; ++kc) {
          if (!mbar_wait(&full_bar[stage], phase, abort_flag)) {
            record_timeout(p.status, abort_flag);
            return false;
          }
          tc_fence_after();
          const uint32_t b_base = smem_u32(sB + stage * S::B_BYTES);
#pragma unroll
          for (int j = 0; j < BK / 16; ++j) {
            const uint64_t adesc = smem_desc_sw128(v_base + kc * (BM * 128) + j * 32, 16, 1024);
            const uint64_t bdesc = B_MN ? smem_desc_sw128(b_base + j * 2048, 8192, 1024)
                                        : smem_desc_sw128(b_base + j * 32, 16, 1024);
            umma_bf16(d, adesc, bdesc, IDESC, (kc > 0 || j > 0) ? 1u : 0u);
          }
          umma_commit(&empty_bar[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        umma_commit(yfull_bar);
        return true;
      };
      for (int tile = range.first; tile < range.end && ok; tile += range.step) {
        const WorkItem item = decode_item<B_RES, CL2>(tile, p, crank);
        const int g = item.g, nt = item.nt, ks0 = item.ks0, ks1 = item.ks1;
        if (B_RES) {
          const int key = g * p.n_tiles + nt;
          if (key != res_key) {
            if (res_loads > 0) umma_commit(bempty_bar);  // old B free after the MMAs so far
            if (!mbar_wait(bfull_bar, res_loads & 1, abort_flag)) {
              record_timeout(p.status, abort_flag);
              ok = false;
              break;
            }
            tc_fence_after();
            res_key = key;
            ++res_loads;
          }
        }
        if (!mbar_wait(&tempty_bar[acc], acc_phase ^ 1, abort_flag)) {
          record_timeout(p.status, abort_flag);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int ks = ks0; ks < ks1; ++ks) {
          if (!mbar_wait(&full_bar[stage], phase, abort_flag)) {
            record_timeout(p.status, abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + stage * S::A_BYTES);
          const uint32_t b_base =
              B_RES ? smem_u32(sRes + ks * S::B_BYTES) : smem_u32(sB + stage * S::B_BYTES);
#pragma unroll
          for (int j = 0; j < BK / 16; ++j) {
            const uint64_t adesc = A_MN ? smem_desc_sw128(a_base + j * 2048, 8192, 1024)
                                        : smem_desc_sw128(a_base + j * 32, 16, 1024);
            const uint64_t bdesc = B_MN ? smem_desc_sw128(b_base + j * 2048, 8192, 1024)
                                        : smem_desc_sw128(b_base + j * 32, 16, 1024);
            umma_bf16(d_tmem, adesc, bdesc, IDESC, (ks > ks0 || j > 0) ? 1u : 0u);
          }
          any_mma = true;
          umma_commit(&empty_bar[stage]);  // frees this smem stage when done
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(&tfull_bar[acc]);  // accumulator ready for the epilogue
        if (EPI == EPI_BLOCK) {
          // block product of the previous tile, into that tile's accumulator
          if (have_prev && !block_mma(tmem_base + static_cast<uint32_t>((acc ^ 1) * BN))) {
            ok = false;
            break;
          }
          have_prev = true;
        }
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      if (EPI == EPI_BLOCK && ok && have_prev &&
          !block_mma(tmem_base + static_cast<uint32_t>((acc ^ 1) * BN)))
        ok = false;
      if (!ok && any_mma) {
        // Wait for the MMAs in flight before TMEM is released.
        umma_commit(drain_bar);
        const unsigned long long t0 = global_timer_ns();
        while (!mbar_try_wait(drain_bar, 0) && global_timer_ns() - t0 < 10000000ull) {
        }
      }
    }
  } else {
    // ----------------------------------------------------------- epilogue
    const int quarter = warp & 3;  // TMEM lanes this warp may read
    uint8_t* stg = sOut + quarter * 4096;
    bool stores_pending = false;
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t yphase = 0;
    bool have_prev = false;  // EPI_BLOCK: a staged tile whose block product is pending
    uint32_t t_prev = 0;
    int prev_row = 0, prev_col0 = 0, prev_acc = 0;
    // EPI_BLOCK: wait for the pending block product, stage it in bf16, free
    // its accumulator and store it as the block output
    auto drain_prev = [&](uint32_t t_src) -> bool {
      const bool ygot = mbar_wait(yfull_bar, yphase, abort_flag);
      yphase ^= 1;
      if (!__all_sync(0xffffffffu, ygot)) {
        record_timeout(p.status, abort_flag);
        return false;
      }
      tc_fence_after();
      if (lane == 0 && stores_pending) bulk_wait_read_all();
      __syncwarp();
      stage_rows_bf16(t_src, sOut, quarter * 32 + lane);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty_bar[prev_acc]);
      fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0) {
        store_staged_rows(&tmY, sOut, quarter, prev_col0, prev_row);
        stores_pending = true;
      }
      return true;
    };
    for (int tile = range.first; tile < range.end; tile += range.step) {
      const WorkItem item = decode_item<B_RES, CL2>(tile, p, crank);
      const int g = item.g, sp = item.sp, mt = item.mt, nt = item.nt;
      const bool got = mbar_wait(&tfull_bar[acc], acc_phase, abort_flag);
      if (!__all_sync(0xffffffffu, got)) {  // the whole warp unwinds together
        record_timeout(p.status, abort_flag);
        break;
      }
      tc_fence_after();
      const uint32_t t_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                              static_cast<uint32_t>(acc * BN);
      if (EPI == EPI_BLOCK) {
        const int out_row = g * p.epi.row_g + sp * p.epi.row_s + mt * BM + quarter * 32;
        const int out_col0 = g * p.epi.col_g + nt * BN;
        // (1) the previous tile's block product: to bf16, free its accumulator, store
        if (have_prev && !drain_prev(t_prev)) break;
        // (2) this tile to bf16 in the staging tile, the A operand of its block
        //     product (issued after the next tile's main loop)
        if (lane == 0 && stores_pending) bulk_wait_read_all();
        __syncwarp();
        stage_rows_bf16(t_base, sOut, quarter * 32 + lane);
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0 && p.store_main) {
          store_staged_rows(&tmC, sOut, quarter, out_col0, out_row);
          stores_pending = true;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(vstaged_bar);
        have_prev = true;
        t_prev = t_base;
        prev_row = out_row;
        prev_col0 = out_col0;
        prev_acc = acc;
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
        continue;  // this accumulator is freed by (1) of the next tile
      } else if (EPI == EPI_ROWS) {
        const int row = mt * BM + quarter * 32 + lane;
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 32) {
          uint32_t r[32];
          tmem_load_32cols(t_base + c0, r);
          tmem_load_wait();
          epilogue_row32(p.epi, g, sp, row, nt * BN + c0, r);
        }
      } else {
        // split item (the last of this CTA): the two CTAs hold the two K halves
        // of one tile; rank r finishes rows 64r .. 64r+63, and the warps with
        // the other half's rows send their partial sums into the peer's ring
        bool send_only = false;
        const uint8_t* recv = nullptr;  // the peer's partial sums (finishing warps)
        const int lr = (quarter & 1) * 32 + lane;  // row within the half
        if (CL2 && item.split) {
          const uint32_t peer = crank ^ 1u;
          // this CTA's MMAs are done and no load follows: its ring is free
          if (quarter == 0 && lane == 0) mbar_arrive_remote(map_peer(smem_u32(xready_bar), peer));
          if ((quarter >> 1) != static_cast<int>(crank)) {
            send_only = true;
            const bool ready = mbar_wait_cluster(xready_bar, 0, abort_flag);
            if (!__all_sync(0xffffffffu, ready)) {
              record_timeout(p.status, abort_flag);
              break;
            }
            const uint32_t dst = map_peer(smem_u32(sA), peer);
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
              uint32_t r[32];
              tmem_load_32cols(t_base + c0, r);
              tmem_load_wait();
#pragma unroll
              for (int i = 0; i < 8; ++i)
                st_cluster_v4(dst + xchg_offset(c0 / 4 + i, lr), r[4 * i], r[4 * i + 1],
                              r[4 * i + 2], r[4 * i + 3]);
            }
            mbar_arrive_remote(map_peer(smem_u32(xfull_bar), peer));
          } else {
            const bool full = mbar_wait_cluster(xfull_bar, 0, abort_flag);
            if (!__all_sync(0xffffffffu, full)) {
              record_timeout(p.status, abort_flag);
              break;
            }
            recv = sA;
          }
        }
        // TMA tile stores: 128-byte rows of 64 bf16 or 32 fp32 per chunk
        constexpr int CW = EPI == EPI_TMA_BF16 ? 64 : 32;
        const int out_row = g * p.epi.row_g + sp * p.epi.row_s + mt * BM + quarter * 32;
        const int out_col0 = g * p.epi.col_g + nt * BN;
        uint8_t* my_row = stg + lane * 128;
#pragma unroll 1
        for (int c0 = 0; c0 < BN && !send_only; c0 += CW) {
          uint32_t w[32];  // this lane's 128 bytes of the chunk
          if (EPI == EPI_TMA_BF16) {
            uint32_t r0[32], r1[32];
            tmem_load_32cols(t_base + c0, r0);
            tmem_load_32cols(t_base + c0 + 32, r1);
            tmem_load_wait();
            if (CL2 && recv != nullptr) {  // + the peer's K half
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float4 a =
                    *reinterpret_cast<const float4*>(recv + xchg_offset(c0 / 4 + i, lr));
                const float4 b =
                    *reinterpret_cast<const float4*>(recv + xchg_offset(c0 / 4 + 8 + i, lr));
                add_f4(r0 + 4 * i, a);
                add_f4(r1 + 4 * i, b);
              }
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              w[j] = pack_bf16x2(r0[2 * j], r0[2 * j + 1]);
              w[16 + j] = pack_bf16x2(r1[2 * j], r1[2 * j + 1]);
            }
          } else {
            tmem_load_32cols(t_base + c0, w);
            tmem_load_wait();
          }
          if (lane == 0 && stores_pending) bulk_wait_read_all();  // staging free again
          __syncwarp();
#pragma unroll
          for (int q = 0; q < 8; ++q)  // 16-byte chunk q of the row, 128B-swizzled
            st_shared_v4(my_row + ((q ^ (lane & 7)) << 4), w[4 * q], w[4 * q + 1], w[4 * q + 2],
                         w[4 * q + 3]);
          fence_proxy_async_shared();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmC, stg, out_col0 + c0, out_row);
            bulk_commit();
            stores_pending = true;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty_bar[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    if (EPI == EPI_BLOCK && have_prev && !*abort_flag) drain_prev(t_prev);
    if (EPI != EPI_ROWS && lane == 0 && stores_pending) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (CL2) cluster_sync();  // no CTA leaves while its peer may still write to it
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, S::TMEM_COLS);
  }
}

// ------------------------------------------------------------- host side

template <bool A_MN, bool B_MN, int BN, bool B_RES, int EPI, bool CL2 = false>
cudaError_t launch_tc(const TcGemm& g, cudaStream_t stream) {
  using S = TcShape<BN, B_RES, EPI>;
  auto* kernel = tc_gemm_kernel<A_MN, B_MN, BN, B_RES, EPI, CL2>;
  // per device, once: the shared-memory attribute and (CL2) the cluster count
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
    if (CL2) {  // clusters of two that fit at once (SMs pair up within a GPC)
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * sm_count());
      cfg.blockDim = dim3(NUM_THREADS);
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
    }
    attr_set[dev] = true;
  }
  const long long cmax = max_clusters[dev];
  lock.unlock();
  CUtensorMap tmA, tmB, tmC, tmR, tmY;
  if (!make_map(&tmA, g.A.ptr, g.A.rows, g.A.cols, g.A.pitch, 2, 64, A_MN ? 64 : BM))
    return cudaErrorInvalidValue;
  // CL2: a K-major B tile is loaded as two halves (one box of BN / 2 rows each)
  if (!make_map(&tmB, g.B.ptr, g.B.rows, g.B.cols, g.B.pitch, 2, 64,
                B_MN ? 64 : (CL2 ? BN / 2 : BN)))
    return cudaErrorInvalidValue;
  if (EPI == EPI_TMA_BF16 || (EPI == EPI_BLOCK && g.epi.out_bf16 != nullptr)) {
    if (!make_map(&tmC, g.epi.out_bf16, g.epi.out_rows, g.epi.ld, g.epi.ld, 2, 64, 32))
      return cudaErrorInvalidValue;
  } else if (EPI == EPI_TMA_F32) {
    if (!make_map(&tmC, g.epi.out_f32, g.epi.out_rows, g.epi.ld, g.epi.ld, 4, 32, 32))
      return cudaErrorInvalidValue;
  } else {
    tmC = tmA;  // unused
  }
  if (EPI == EPI_BLOCK) {
    if (g.epi.out_bf16 == nullptr) tmC = tmA;  // no main output: never stored
    if (!make_map(&tmR, g.blk.ptr, g.blk.rows, g.blk.cols, g.blk.pitch, 2, 64, B_MN ? 64 : BN))
      return cudaErrorInvalidValue;
    if (!make_map(&tmY, g.out_blk, g.epi.out_rows, g.epi.ld, g.epi.ld, 2, 64, 32))
      return cudaErrorInvalidValue;
  } else {
    tmR = tmA;  // unused
    tmY = tmA;
  }

  TcKernelArgs p;
  p.m_tiles = (g.M + BM - 1) / BM;
  p.m_pairs = (p.m_tiles + 1) / 2;
  p.tail_first = p.items = p.k_half = 0;  // set for CL2 below
  p.n_tiles = g.N / BN;
  p.k_steps_total = (g.K + BK - 1) / BK;
  const int splits = tc_effective_splits(g.K, g.splits);
  p.k_steps_per_split = (p.k_steps_total + splits - 1) / splits;
  p.splits = splits;
  p.batches = g.batches;
  p.a_mn_per_g = g.A.mn_per_g;
  p.a_k_per_g = g.A.k_per_g;
  p.b_mn_per_g = g.B.mn_per_g;
  p.b_k_per_g = g.B.k_per_g;
  p.epi = g.epi;
  p.store_main = g.epi.out_bf16 != nullptr ? 1 : 0;
  p.status = device_status_ptr();
  if (B_RES && (p.splits != 1 || p.k_steps_total > S::MAX_RES_KSTEPS))
    return cudaErrorInvalidValue;
  if (CL2) {
    const long long units =
        static_cast<long long>(p.batches) * p.splits * p.m_pairs * p.n_tiles;
    if (units <= 0) return cudaSuccess;
    int clusters = static_cast<int>(std::min<long long>(units, cmax));
    // A last round of r < cmax units leaves clusters idle; when 2r fit in one
    // round, its 2r tiles go to 2r clusters instead, each tile's K steps
    // split between the cluster's two CTAs (half the round's time).
    p.tail_first = static_cast<int>(units);
    p.items = static_cast<int>(units);
    p.k_half = p.k_steps_total / 2;
    if (g.split_tail && p.batches == 1 && p.splits == 1 && p.k_steps_total % 2 == 0) {
      const long long r = units % cmax;
      if (units >= cmax && r > 0 && 2 * r <= cmax) {
        p.tail_first = static_cast<int>(units - r);
        p.items = static_cast<int>(units + r);
      } else if (units < cmax && 2 * units <= cmax) {
        p.tail_first = 0;
        p.items = static_cast<int>(2 * units);
        clusters = static_cast<int>(2 * units);
      }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(NUM_THREADS);
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
  const long long tiles = static_cast<long long>(p.batches) * p.splits * p.m_tiles * p.n_tiles;
  if (tiles <= 0) return cudaSuccess;
  int grid = static_cast<int>(std::min<long long>(tiles, sm_count()));
  if (B_RES) {  // contiguous runs: launch only the CTAs that get a run
    const long long per = (tiles + grid - 1) / grid;
    grid = static_cast<int>((tiles + per - 1) / per);
  }
  prof_begin(g.tag, stream);
  cudaError_t e = launch_pdl(kernel, dim3(grid), dim3(NUM_THREADS), S::SMEM, stream, tmA, tmB,
                             tmC, tmR, tmY, p);
  prof_end(g.tag, stream);
  return e != cudaSuccess ? e : cudaGetLastError();
}

bool plain_output(const EpiArgs& e) {
  return e.alpha == 1.f && e.X == nullptr && e.Y == nullptr && e.delta == 0.f &&
         ((e.out_f32 == nullptr) != (e.out_bf16 == nullptr)) && e.out_rows > 0;
}

}  // namespace

int tc_effective_splits(int K, int want) {
  const int ksteps = (K + BK - 1) / BK;
  int splits = std::max(1, std::min(want, ksteps));
  const int per = (ksteps + splits - 1) / splits;
  return (ksteps + per - 1) / per;  // no empty split
}

cudaError_t tc_gemm_run(const TcGemm& g, cudaStream_t stream) {
  if (g.M <= 0 || g.N <= 0 || g.K <= 0 || g.batches <= 0) return cudaSuccess;
  if ((g.BN != 128 && g.BN != 256) || g.N % g.BN != 0) return cudaErrorInvalidValue;
  const bool a = g.A.mn_major, b = g.B.mn_major;
  if (g.out_blk != nullptr) {
    // W0 GEMM with the block-diagonal factor applied in its epilogue; the
    // block operand has the same major-ness as B
    if (g.BN != 256 || g.b_resident || a || g.batches != 1 || g.splits != 1 ||
        g.blk.mn_major != b || g.epi.out_f32 != nullptr || g.epi.alpha != 1.f ||
        g.epi.X != nullptr || g.epi.Y != nullptr || g.epi.delta != 0.f || g.epi.out_rows <= 0)
      return cudaErrorInvalidValue;
    if (!b) return launch_tc<false, false, 256, false, EPI_BLOCK>(g, stream);
    return launch_tc<false, true, 256, false, EPI_BLOCK>(g, stream);
  }
  if (!plain_output(g.epi)) {
    // general epilogue: the b x b products of the block build and its adjoint
    if (g.BN != 128 || g.b_resident) return cudaErrorInvalidValue;
    if (!a && !b) return launch_tc<false, false, 128, false, EPI_ROWS>(g, stream);
    if (!a && b) return launch_tc<false, true, 128, false, EPI_ROWS>(g, stream);
    if (a && b) return launch_tc<true, true, 128, false, EPI_ROWS>(g, stream);
    return cudaErrorInvalidValue;
  }
  const bool bf16_out = g.epi.out_bf16 != nullptr;
  if (g.b_resident) {  // block-diagonal transforms (bf16 out)
    if (a || !bf16_out) return cudaErrorInvalidValue;
    if (g.BN == 256) {
      if (!b) return launch_tc<false, false, 256, true, EPI_TMA_BF16>(g, stream);
      return launch_tc<false, true, 256, true, EPI_TMA_BF16>(g, stream);
    }
    if (!b) return launch_tc<false, false, 128, true, EPI_TMA_BF16>(g, stream);
    return launch_tc<false, true, 128, true, EPI_TMA_BF16>(g, stream);
  }
  if (g.BN != 256) return cudaErrorInvalidValue;
  if (bf16_out) {  // the W0 GEMM and its transpose
    if (g.cluster2 && g.batches == 1 && g.splits == 1 && g.M > BM) {  // B shared by two CTAs
      if (!a && !b) return launch_tc<false, false, 256, false, EPI_TMA_BF16, true>(g, stream);
      if (!a && b) return launch_tc<false, true, 256, false, EPI_TMA_BF16, true>(g, stream);
    }
    if (!a && !b) return launch_tc<false, false, 256, false, EPI_TMA_BF16>(g, stream);
    if (!a && b) return launch_tc<false, true, 256, false, EPI_TMA_BF16>(g, stream);
    return cudaErrorInvalidValue;
  }
  // per-block sums over tokens (fp32 split-K partials)
  if (a && b) return launch_tc<true, true, 256, false, EPI_TMA_F32>(g, stream);
  return cudaErrorInvalidValue;
}

}  // namespace poetx
