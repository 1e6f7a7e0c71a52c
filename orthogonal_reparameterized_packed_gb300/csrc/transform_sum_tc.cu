// The backward's two passes over one activation gradient fused into one
// kernel (sm_103a, tcgen05 + TMA): for a gradient X [T][d], another
// activation Z [T][d] and the 256 x 256 superblocks SB of one side,
//
//   out[t][g*256 + n]  = sum_kk X[t][g*256 + kk] SB[g*256 + kk][n]     (bf16)
//   part[s][g][m][n]   = sum_{t in split s} Z[t][g*256 + m] X[t][g*256 + n]  (fp32)
//
// i.e. the transposed block transform (dv = dy R, dx = du P) and the
// split-K token sums G^T of the block gradients (sum_t v_t dy_t^T,
// sum_t x_t du_t^T).  Separately they read X twice from HBM; here every X
// tile that lands in shared memory feeds both products.
//
// One CTA per (block g, half h, token split s):
//   transform half: out columns g*256 + h*128 .. +127, all 256 K features;
//                   SB's 256 x 128 half stays resident in shared memory
//   sum half:       rows m = h*128 .. +127 of part[s][g], all 256 columns
// Both halves of a block read the same X tiles at about the same time, so
// the second read is served by L2.  TMEM: two 128-column accumulators for
// the transform tiles (the epilogue of one overlaps the next) and one
// 256-column accumulator for the sum, 512 columns in all.
//
// Warp roles: warp 0 TMA producer, warp 1 TMEM owner + transform MMA issuer,
// warp 6 token-sum MMA issuer, warps 2-5 epilogue (transform tiles: row-per-thread 16-byte stores, as the shared
// memory a TMA-store staging tile would take holds two more gradient chunks
// in flight; the split's partial sum at the end: staged in the then idle
// operand rings and stored by TMA).  Every wait is bounded; on expiry the CTA
// records POETX_ERR_TIMEOUT, lets its copies and MMAs in flight land and
// returns.
#include <algorithm>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace poetx {

namespace {

constexpr int TS_THREADS = 224;
constexpr int TS_XSTAGES = 6;                  // X ring: one 128 x 64 chunk per stage
// a tile's chunk pairs (0,1), (2,3) sit in adjacent slots (2i, 2i+1): tiles
// start on even slots when the ring length is even
static_assert(TS_XSTAGES % 2 == 0, "even ring length");
constexpr int TS_ZSTAGES = 2;                  // Z ring: one 128 x 128 half tile per stage
constexpr int TS_RES_BYTES = 256 * 128 * 2;    // SB half, 64 KiB
constexpr int TS_X_BYTES = BM * 64 * 2;        // 16 KiB
constexpr int TS_Z_BYTES = BM * 128 * 2;       // 32 KiB
constexpr int TS_BAR_BYTES = 256;
constexpr int TS_SMEM =
    1024 + TS_RES_BYTES + TS_XSTAGES * TS_X_BYTES + TS_ZSTAGES * TS_Z_BYTES + TS_BAR_BYTES;
constexpr uint32_t TS_TMEM_COLS = 512;
static_assert(TS_SMEM <= 227 * 1024, "shared memory per CTA");
static_assert((2 * TS_XSTAGES + 2 * TS_ZSTAGES + 4 + 2 + 2) * 8 + 8 <= TS_BAR_BYTES,
              "barriers exceed their shared-memory area");
// the final partial sum is staged in the idle X and Z rings: 4 warps x 32 KiB
static_assert(TS_XSTAGES * TS_X_BYTES + TS_ZSTAGES * TS_Z_BYTES >= 4 * 32768, "staging room");

struct TsArgs {
  int d;            // features (multiple of 256)
  int m_tiles;      // token tiles of 128
  int splits;       // token splits
  int per;          // token tiles per split
  long long T;      // tokens
  __nv_bfloat16* out;  // [T][d]
  float* part;         // [splits][d][256]
  int* status;
};

__global__ void __launch_bounds__(TS_THREADS, 1)
    transform_sum_kernel(const __grid_constant__ CUtensorMap tmX,   // X [T][d], box 64 x 128
                         const __grid_constant__ CUtensorMap tmZ,   // Z [T][d], box 64 x 128
                         const __grid_constant__ CUtensorMap tmB,   // SB [d][256], box 64 x 64
                         const __grid_constant__ CUtensorMap tmP,   // part [splits*d][256] fp32, box 32 x 32
                         const TsArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sRes = base;
  uint8_t* sX = sRes + TS_RES_BYTES;
  uint8_t* sZ = sX + TS_XSTAGES * TS_X_BYTES;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(sZ + TS_ZSTAGES * TS_Z_BYTES);
  uint64_t* empty_bar = full_bar + TS_XSTAGES;
  uint64_t* zfull_bar = empty_bar + TS_XSTAGES;
  uint64_t* zempty_bar = zfull_bar + TS_ZSTAGES;
  uint64_t* tfull_bar = zempty_bar + TS_ZSTAGES;  // [2]
  uint64_t* tempty_bar = tfull_bar + 2;           // [2]
  uint64_t* bfull_bar = tempty_bar + 2;
  uint64_t* gfull_bar = bfull_bar + 1;
  uint64_t* drain_bar = gfull_bar + 1;   // [2]: one per MMA issuer
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  // work unit: token split fastest, then the half, then the block
  const int s = blockIdx.x % p.splits;
  const int h = (blockIdx.x / p.splits) & 1;
  const int g = blockIdx.x / (2 * p.splits);
  const int t_first = s * p.per;
  const int t_end = min(t_first + p.per, p.m_tiles);
  const int col_blk = g * 256;

  if (threadIdx.x == 0) {
    for (int i = 0; i < TS_XSTAGES; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 2);  // released by both MMA issuers
    }
    for (int i = 0; i < TS_ZSTAGES; ++i) {
      mbar_init(&zfull_bar[i], 1);
      mbar_init(&zempty_bar[i], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], 4);
    }
    mbar_init(bfull_bar, 1);
    mbar_init(gfull_bar, 1);
    mbar_init(&drain_bar[0], 1);
    mbar_init(&drain_bar[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmZ);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmP);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, TS_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  pdl_trigger();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ TMA producer
      bool ok = true;
      int xs = 0, zs = 0;
      uint32_t xphase = 0, zphase = 0;
      long long x_issued = 0, z_issued = 0;
      // SB's half: K rows g*256 .. +255, columns h*128 .. +127 (MN-major B)
      mbar_arrive_expect_tx(bfull_bar, TS_RES_BYTES);
      for (int kc = 0; kc < 4; ++kc)
        for (int c2 = 0; c2 < 2; ++c2)
          tma_load_2d(sRes + kc * 16384 + c2 * 8192, &tmB, bfull_bar, h * 128 + 64 * c2,
                      col_blk + kc * 64);
      for (int t = t_first; t < t_end && ok; ++t) {
        if (!mbar_wait(&zempty_bar[zs], zphase ^ 1, abort_flag)) {
          record_timeout(p.status, abort_flag);
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&zfull_bar[zs], TS_Z_BYTES);
        uint8_t* z_dst = sZ + zs * TS_Z_BYTES;
        tma_load_2d(z_dst, &tmZ, &zfull_bar[zs], col_blk + h * 128, t * BM);
        tma_load_2d(z_dst + 16384, &tmZ, &zfull_bar[zs], col_blk + h * 128 + 64, t * BM);
        ++z_issued;
        if (++zs == TS_ZSTAGES) {
          zs = 0;
          zphase ^= 1;
        }
        for (int c = 0; c < 4; ++c) {
          if (!mbar_wait(&empty_bar[xs], xphase ^ 1, abort_flag)) {
            record_timeout(p.status, abort_flag);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full_bar[xs], TS_X_BYTES);
          tma_load_2d(sX + xs * TS_X_BYTES, &tmX, &full_bar[xs], col_blk + 64 * c, t * BM);
          ++x_issued;
          if (++xs == TS_XSTAGES) {
            xs = 0;
            xphase ^= 1;
          }
        }
      }
      if (!ok) {  // let the copies in flight land before the CTA exits
        auto settle = [](uint64_t* bars, int nst, int st, uint32_t ph, long long issued) {
          const int outstanding = issued < nst ? static_cast<int>(issued) : nst;
          for (int i = 0; i < outstanding; ++i) {
            if (--st < 0) {
              st = nst - 1;
              ph ^= 1;
            }
            const unsigned long long t0 = global_timer_ns();
            while (!mbar_try_wait(&bars[st], ph) && global_timer_ns() - t0 < 10000000ull) {
            }
          }
        };
        settle(full_bar, TS_XSTAGES, xs, xphase, x_issued);
        settle(zfull_bar, TS_ZSTAGES, zs, zphase, z_issued);
        const unsigned long long t0 = global_timer_ns();
        while (!mbar_try_wait(bfull_bar, 0) && global_timer_ns() - t0 < 10000000ull) {
        }
      }
    }
  } else if (warp == 1 || warp == 6) {
    if (lane == 0) {
      // ------------------------------------------------------ MMA issuers
      // Warp 1 issues the transform tiles (into the two rotating
      // accumulators), warp 6 the token sums (into the persistent one): two
      // threads keep the tensor pipe fed through each other's barrier waits.
      // An X slot is free once both have committed it.
      const bool sums = warp == 6;
      constexpr uint32_t IDESC_T = instr_desc_bf16(BM, 128, false, true);  // X K-major, SB MN-major
      constexpr uint32_t IDESC_S = instr_desc_bf16(BM, 128, true, true);   // Z, X both MN-major
      const uint32_t g_tmem = tmem_base + 256u;
      uint64_t* my_drain = &drain_bar[sums ? 1 : 0];
      bool ok = sums || mbar_wait(bfull_bar, 0, abort_flag);  // SB: transforms only
      if (!ok) record_timeout(p.status, abort_flag);
      tc_fence_after();
      bool any_mma = false;
      int xs = 0, zs = 0, acc = 0;
      uint32_t xphase = 0, zphase = 0, acc_phase = 0;
      const uint32_t res_base = smem_u32(sRes);
      for (int t = t_first; t < t_end && ok; ++t) {
        const bool ready = sums ? mbar_wait(&zfull_bar[zs], zphase, abort_flag)
                                : mbar_wait(&tempty_bar[acc], acc_phase ^ 1, abort_flag);
        if (!ready) {
          record_timeout(p.status, abort_flag);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t t_tmem = tmem_base + static_cast<uint32_t>(acc * 128);
        const uint32_t z_base = smem_u32(sZ + zs * TS_Z_BYTES);
        for (int c = 0; c < 4; ++c) {
          if (!mbar_wait(&full_bar[xs], xphase, abort_flag)) {
            record_timeout(p.status, abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t x_base = smem_u32(sX + xs * TS_X_BYTES);
          if (!sums) {
            // transform: out tile += X chunk c (K = features 64c ..) x SB rows 64c ..
#pragma unroll
            for (int j = 0; j < 4; ++j)
              umma_bf16(t_tmem, smem_desc_sw128(x_base + j * 32, 16, 1024),
                        smem_desc_sw128(res_base + c * 16384 + j * 2048, 8192, 1024), IDESC_T,
                        (c > 0 || j > 0) ? 1u : 0u);
            umma_commit(&empty_bar[xs]);
            any_mma = true;
          } else if (c & 1) {
            // token sum over chunks c-1, c (adjacent ring slots: a tile's chunk
            // i always sits in slot i): G[m][64(c-1) ..] += sum_t Z[t][m] X[t][..]
            const uint32_t x_pair = x_base - TS_X_BYTES;
#pragma unroll
            for (int j = 0; j < 8; ++j)
              umma_bf16(g_tmem + static_cast<uint32_t>(64 * (c - 1)),
                        smem_desc_sw128(z_base + j * 2048, 16384, 1024),
                        smem_desc_sw128(x_pair + j * 2048, TS_X_BYTES, 1024), IDESC_S,
                        (t > t_first || j > 0) ? 1u : 0u);
            umma_commit(&empty_bar[xs - 1]);
            umma_commit(&empty_bar[xs]);
            any_mma = true;
          }
          if (++xs == TS_XSTAGES) {
            xs = 0;
            xphase ^= 1;
          }
        }
        if (!ok) break;
        if (!sums) {
          umma_commit(&tfull_bar[acc]);
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1;
        } else {
          umma_commit(&zempty_bar[zs]);
          if (++zs == TS_ZSTAGES) {
            zs = 0;
            zphase ^= 1;
          }
        }
      }
      if (ok) {
        if (sums) umma_commit(gfull_bar);  // the split's sum is complete
      } else if (any_mma) {
        umma_commit(my_drain);
        const unsigned long long t0 = global_timer_ns();
        while (!mbar_try_wait(my_drain, 0) && global_timer_ns() - t0 < 10000000ull) {
        }
      }
    }
  } else {
    // ----------------------------------------------------------- epilogue
    // Each thread owns one accumulator row and stores it with 16-byte stores
    // (the transform tile's 128 bf16 columns, then the sum's 256 fp32).
    const int quarter = warp & 3;
    const int row_in_tile = quarter * 32 + lane;
    bool ok = true;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = t_first; t < t_end; ++t) {
      const bool got = mbar_wait(&tfull_bar[acc], acc_phase, abort_flag);
      if (!__all_sync(0xffffffffu, got)) {
        record_timeout(p.status, abort_flag);
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t t_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                              static_cast<uint32_t>(acc * 128);
      const long long row = static_cast<long long>(t) * BM + row_in_tile;
      uint4* dst = reinterpret_cast<uint4*>(p.out + row * p.d + col_blk + h * 128);
#pragma unroll 1
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t r[32];
        tmem_load_32cols(t_base + c0, r);
        tmem_load_wait();
        if (row < p.T) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            dst[c0 / 8 + q] = make_uint4(pack_bf16x2(r[8 * q], r[8 * q + 1]),
                                         pack_bf16x2(r[8 * q + 2], r[8 * q + 3]),
                                         pack_bf16x2(r[8 * q + 4], r[8 * q + 5]),
                                         pack_bf16x2(r[8 * q + 6], r[8 * q + 7]));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty_bar[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    if (ok && t_end > t_first) {
      // the split's partial sum: rows h*128 + 32*quarter .. of part[s][g], fp32.
      // Once the last MMA is done the operand rings are idle: each warp stages
      // its 32 rows there as eight 128B-swizzled 32 x 32 boxes (32 KiB per
      // warp, 128 KiB in all across the X and Z rings) and stores them by TMA.
      const bool got = mbar_wait(gfull_bar, 0, abort_flag);
      if (!__all_sync(0xffffffffu, got)) {
        record_timeout(p.status, abort_flag);
      } else {
        tc_fence_after();
        const uint32_t g_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + 256u;
        uint8_t* stg = sX + quarter * 32768;
#pragma unroll 1
        for (int cc = 0; cc < 8; ++cc) {
          uint32_t r[32];
          tmem_load_32cols(g_base + cc * 32, r);
          tmem_load_wait();
          uint8_t* row = stg + cc * 4096 + lane * 128;
#pragma unroll
          for (int q = 0; q < 8; ++q)
            st_shared_v4(row + ((q ^ (lane & 7)) << 4), r[4 * q], r[4 * q + 1], r[4 * q + 2],
                         r[4 * q + 3]);
        }
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) {
          const int prow0 = s * p.d + col_blk + h * 128 + quarter * 32;
#pragma unroll 1
          for (int cc = 0; cc < 8; ++cc) tma_store_2d(&tmP, stg + cc * 4096, cc * 32, prow0);
          bulk_commit();
          bulk_wait_all();
        }
        __syncwarp();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, TS_TMEM_COLS);
  }
}

}  // namespace

// Token splits: one CTA per (block, half, split) and one CTA per SM, so the
// launch runs in ceil(CTAs / SMs) waves of `per` token tiles each.  The
// split count minimises waves x (per + 3), the 3 standing for a CTA's fixed
// cost in tile times (the pipeline fill, the resident block half in, the
// partial sum out); more splits are taken only for a gain of over 5 %
// (they add partial sums to add up).  One wave where one fits (d = 4096,
// 16384 tokens: 4 splits, 128 CTAs); wide sides take several (d = 14336:
// 4 splits in 3 waves instead of 112 CTAs over the whole run).
int transform_sum_splits(int d, long long T) {
  const int m_tiles = static_cast<int>((T + BM - 1) / BM);
  const int units = 2 * (d / 256);
  if (m_tiles <= 1 || units <= 0) return 1;
  const long long sms = sm_count();
  int best = 1;
  long long best_cost = -1;
  const int max_splits = static_cast<int>(std::min<long long>(m_tiles, 2 * sms));
  for (int s = 1; s <= max_splits; ++s) {
    const int per = (m_tiles + s - 1) / s;
    if ((m_tiles + per - 1) / per != s) continue;  // no empty split
    const long long waves = (static_cast<long long>(units) * s + sms - 1) / sms;
    const long long cost = waves * (per + 3);
    if (best_cost < 0 || cost * 20 < best_cost * 19) {
      best = s;
      best_cost = cost;
    }
  }
  return best;
}

cudaError_t tc_transform_sum(const __nv_bfloat16* X, const __nv_bfloat16* Z,
                             const __nv_bfloat16* sb, __nv_bfloat16* out, float* part, int d,
                             long long T, int splits, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  if (d <= 0 || d % 256 != 0 || splits != transform_sum_splits(d, T)) return cudaErrorInvalidValue;
  static bool attr_set[64] = {false};
  static std::mutex mu;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_set[dev]) {
      cudaError_t e = cudaFuncSetAttribute(transform_sum_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, TS_SMEM);
      if (e != cudaSuccess) return e;
      attr_set[dev] = true;
    }
  }
  CUtensorMap tmX, tmZ, tmB, tmP;
  if (!make_map(&tmX, X, T, d, d, 2, 64, BM) || !make_map(&tmZ, Z, T, d, d, 2, 64, BM) ||
      !make_map(&tmB, sb, d, 256, 256, 2, 64, 64) ||
      !make_map(&tmP, part, static_cast<long long>(splits) * d, 256, 256, 4, 32, 32))
    return cudaErrorInvalidValue;
  if (reinterpret_cast<uintptr_t>(out) % 16 != 0 || reinterpret_cast<uintptr_t>(part) % 16 != 0)
    return cudaErrorInvalidValue;
  TsArgs a;
  a.d = d;
  a.m_tiles = static_cast<int>((T + BM - 1) / BM);
  a.splits = splits;
  a.per = (a.m_tiles + splits - 1) / splits;
  a.T = T;
  a.out = out;
  a.part = part;
  a.status = device_status_ptr();
  const int grid = 2 * (d / 256) * splits;
  prof_begin("transform_sum", stream);
  cudaError_t e = launch_pdl(transform_sum_kernel, dim3(grid), dim3(TS_THREADS), TS_SMEM, stream,
                             tmX, tmZ, tmB, tmP, a);
  prof_end("transform_sum", stream);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace poetx
