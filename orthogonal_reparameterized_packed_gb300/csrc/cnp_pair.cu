// The Cayley-Neumann block build for k = 3 on CTA pairs, every operand in
// shared memory: the pages' fused CNP kernel that loads Q (and Q^2) into
// shared memory once, laid out for two SMs.
//
// One cluster of two CTAs per 256 x 256 superblock (one block of b = 256, or
// 256 / b blocks of b = 32, 64, 128 on its diagonal: products of block-
// diagonal matrices stay block diagonal).  CTA rank r owns rows 128 r ..
// 128 r + 127 of every matrix; a pair MMA (M = 256 over both CTAs, N = 256,
// D = A B^T) reads A from each CTA's own rows and B from each CTA's own
// rows of the second operand, so with Q^T = -Q and (Q^2)^T = Q^2 no matrix
// ever has to be transposed or exchanged:
//
//   R = I + 2Q + 2Q^2 + 2Q^3 + Q^4 = I + 2Q + 2 Q2 + Q2 W^T,
//   Q2 = Q Q = -(Q Q^T),  W = Q2 - 2Q  (W^T = Q2 + 2Q)
//
//   prologue  theta -> Q as bf16 hi + lo parts (own rows, both triangles;
//             the packed rows staged in shared memory by bulk copies)
//   phase 1   acc0 = Q Q^T                              (16 pair MMAs)
//   epilogue  Q2 = -acc0 -> bf16; W = Q2 - 2Q -> bf16;
//             acc0 <- I + 2Q + 2 Q2 in fp32 (2Q exact from hi + lo)
//   phase 2   acc1 = Q2 W^T                             (16 pair MMAs)
//   epilogue  block rows = acc0 + acc1 -> bf16 (the diagonal b-blocks)
//
// Shared memory per CTA: three 128 x 256 bf16 operand tiles (Q hi, later
// W; Q2; Q lo), each four 128B-swizzled K-major 128 x 64 chunks.  TMEM: two
// 256-column fp32 accumulators.  Every wait is bounded; on expiry the CTA
// records POETX_ERR_TIMEOUT and leaves through the final cluster barrier.
#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace poetx {

namespace {

// Ten warps: warp 1 holds TMEM (and in the leader issues the MMAs); warps
// 2..9 run the epilogues, two per TMEM lane quarter, each on half of the
// columns; all ten unpack the parameters in the prologue.
constexpr int kCnpThreads = 320;
constexpr int kOpBytes = BM * 256 * 2;  // one operand tile: 128 rows x 256 columns bf16
// The prologue stages the packed parameters it reads in the (not yet used)
// Q2 tile and an extra 32 KiB behind it: at most the strict upper triangle's
// rows 0..127 of a 256-block, 24512 floats = 98048 bytes.
constexpr int kStageBytes = kOpBytes + 32768;
constexpr int kBuildSmem = 1024 + 2 * kOpBytes + kStageBytes + 256;
static_assert(kBuildSmem <= 227 * 1024, "shared memory per CTA");
static_assert(kStageBytes >= (32640 - 8128) * 4, "staging for rows 0..127 of a 256-block");

// Byte offset of element (row, col) of an operand tile: chunk col / 64,
// 128-byte row, 16-byte group (col % 64) / 8 swizzled with row % 8.
__device__ __forceinline__ uint32_t op_off(int row, int col) {
  return static_cast<uint32_t>((col >> 6) * (BM * 128) + row * 128 +
                               ((((col & 63) >> 3) ^ (row & 7)) << 4) + ((col & 7) << 1));
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// D (+)= A B^T over K = 256 for two operand tiles (both K-major), pair MMA.
__device__ __forceinline__ void mma_tiles(uint32_t d_tmem, const uint8_t* A, const uint8_t* B,
                                          uint32_t idesc) {
  const uint32_t a0 = smem_u32(A), b0 = smem_u32(B);
#pragma unroll
  for (int kc = 0; kc < 4; ++kc)
#pragma unroll
    for (int j = 0; j < BK / 16; ++j)
      umma_bf16_pair(d_tmem, smem_desc_sw128(a0 + kc * (BM * 128) + j * 32, 16, 1024),
                     smem_desc_sw128(b0 + kc * (BM * 128) + j * 32, 16, 1024), idesc,
                     (kc > 0 || j > 0) ? 1u : 0u);
}

struct CnpBuildArgs {
  const float* theta;    // [n][b(b-1)/2]
  int b, nb;             // block size, blocks per superblock (256 / b)
  __nv_bfloat16* blocks; // [n][b][b]
  int* status;
};

__global__ void __launch_bounds__(kCnpThreads, 1) cnp_build_pair_kernel(const CnpBuildArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* tA = base;                 // Q hi, then W
  uint8_t* tC = base + kOpBytes;      // Q lo
  uint8_t* tB = base + 2 * kOpBytes;  // staged theta, then Q2
  uint64_t* ready1 = reinterpret_cast<uint64_t*>(base + 2 * kOpBytes + kStageBytes);
  uint64_t* p1done = ready1 + 1;  // each CTA: phase-1 MMAs done
  uint64_t* ready2 = p1done + 1;  // leader: Q2, W written (eight warps of each CTA)
  uint64_t* p2done = ready2 + 1;  // each CTA: phase-2 MMAs done
  uint64_t* drain = p2done + 1;
  uint64_t* staged = drain + 1;  // the bulk copy of theta has landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(staged + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int rank = static_cast<int>(cluster_ctarank());
  const bool leader = rank == 0;
  const int sb = static_cast<int>(cluster_id_x());
  const int b = a.b;

  if (threadIdx.x == 0) {
    mbar_init(ready1, 2);
    mbar_init(p1done, 1);
    mbar_init(ready2, 16);
    mbar_init(p2done, 1);
    mbar_init(drain, 1);
    mbar_init(staged, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  pdl_trigger();

  // ---------------------------------------------------------------- prologue
  // The packed rows this CTA reads: b = 256: rank 0 the triangle's rows
  // 0..127, rank 1 its rows 128..254 (each a contiguous range); b <= 128:
  // the whole triangles of the blocks in this CTA's half.  Bulk copies
  // bring them into shared memory (the Q2 tile, not yet in use).
  const int P = b * (b - 1) / 2;
  const int lb = __ffs(b) - 1;  // b is a power of two
  const int bl0 = b <= 128 ? rank * (a.nb / 2) : 0;
  const int nbl = b <= 128 ? a.nb / 2 : 1;
  const int row0 = b <= 128 ? 0 : 128 * rank;           // first staged triangle row
  const int row1 = b <= 128 ? b - 1 : 128 * rank + 128;  // one past the last
  auto tri_start = [&](int ib) { return ib * b - ib * (ib + 1) / 2; };
  const int s0 = tri_start(row0);
  const int per_block = (row1 >= b - 1 ? P : tri_start(row1)) - s0;  // floats staged per block
  const float* src = a.theta + (static_cast<long long>(sb) * a.nb + bl0) * P + s0;
  const uint32_t stage_bytes = static_cast<uint32_t>(nbl * per_block) * 4u;
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(staged, stage_bytes);
    // 16-byte aligned: P * 4 and tri_start(128) * 4 (256-blocks) are multiples of 16
    for (uint32_t off = 0; off < stage_bytes; off += 32768u)
      bulk_load_1d(tB + off, reinterpret_cast<const uint8_t*>(src) + off,
                   stage_bytes - off < 32768u ? stage_bytes - off : 32768u, staged);
  }
  {
    // Every 8-column group of this CTA's tiles is written once:
    // Q[p][c] = +theta(p, c) (c > p: staged row p), -theta(c, p) (c < p:
    // staged row c), 0 on the diagonal and outside the diagonal b-blocks.
    // For b = 256 the columns 0..127 of rank 1's rows come from rows
    // 0..127 of the triangle, which rank 0 staged: rank 1 reads those from
    // rank 0's shared memory.  Items run rows fastest, so a warp covers 32
    // rows of one group: the same branch for almost every lane, and the
    // lower-triangle reads of consecutive rows are consecutive words.
    const bool got = mbar_wait(staged, 0, abort_flag);
    if (!got) record_timeout(a.status, abort_flag);
    if (b == 256) cluster_sync();  // rank 0's staging has landed before rank 1 reads it
    const float* st = reinterpret_cast<const float*>(tB);
    const uint32_t peer_st = map_peer(smem_u32(tB), 0);  // rank 0's staging (b = 256)
    const int lg = lb - 3;  // log2 of the 8-column groups per block row
    if (b <= 128) {  // zeros outside the blocks: 32 - b/8 groups of each row
      const int zg = 32 - (b >> 3);
      for (int t = threadIdx.x; got && t < 128 * zg; t += kCnpThreads) {
        const int row = t & 127, k = t >> 7;
        const int p = 128 * rank + row;
        const int own0 = (p >> lb) << lg;  // first group of the row's block
        const int g = k < own0 ? k : k + (b >> 3);
        const uint32_t off = op_off(row, 8 * g);
        st_shared_v4(tA + off, 0u, 0u, 0u, 0u);
        st_shared_v4(tC + off, 0u, 0u, 0u, 0u);
      }
    }
    const int groups = b <= 128 ? (b >> 3) : 32;  // in-block groups per row
    for (int t = threadIdx.x; got && t < 128 * groups; t += kCnpThreads) {
      const int row = t & 127;
      const int p = 128 * rank + row;
      const int blk = p >> lb;
      const int c8 = (blk << lb) + 8 * (t >> 7);
      const int pb = p - (blk << lb), cb = c8 - (blk << lb);  // in-block row, first column
      const float* sblk = st + (blk - bl0) * per_block - s0;  // + tri_start(row) + ...
      float v[8];
      if (cb > pb) {  // upper: row pb of the triangle, entries cb - pb - 1 ..
        const float* r = sblk + tri_start(pb) + (cb - pb - 1);
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = r[e];
      } else if (cb + 7 < pb) {  // lower: -theta(c, p) from rows c = cb .. cb + 7
        int at = tri_start(cb) + (pb - cb - 1);
        if (b == 256 && rank == 1 && cb < 128) {  // rows c < 128: rank 0's staging
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            v[e] = -ld_cluster_f32(peer_st + 4u * static_cast<uint32_t>(at));
            at += b - (cb + e) - 2;  // tri_start(c + 1) - tri_start(c) - 1
          }
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            v[e] = -sblk[at];
            at += b - (cb + e) - 2;
          }
        }
      } else {  // the group holding the diagonal (never in rank 1's columns < 128)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int c = cb + e;
          v[e] = c > pb ? sblk[tri_start(pb) + (c - pb - 1)]
                        : (c < pb ? -sblk[tri_start(c) + (pb - c - 1)] : 0.f);
        }
      }
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const __nv_bfloat162 hi = __floats2bfloat162_rn(v[e], v[e + 1]);
        const __nv_bfloat162 lo = __floats2bfloat162_rn(v[e] - __low2float(hi),
                                                        v[e + 1] - __high2float(hi));
        hw[e / 2] = *reinterpret_cast<const uint32_t*>(&hi);
        lw[e / 2] = *reinterpret_cast<const uint32_t*>(&lo);
      }
      const uint32_t off = op_off(row, c8);
      st_shared_v4(tA + off, hw[0], hw[1], hw[2], hw[3]);
      st_shared_v4(tC + off, lw[0], lw[1], lw[2], lw[3]);
    }
  }
  fence_proxy_async_all();  // generic writes (here and in the peer) -> the tensor cores' reads
  cluster_sync();           // both CTAs' tiles are complete
  if (threadIdx.x == 0) mbar_arrive_remote(map_peer(smem_u32(ready1), 0));

  constexpr uint32_t IDESC = instr_desc_bf16(2 * BM, 256, false, false);
  if (warp == 1) {
    if (lane == 0 && leader) {
      // ----------------------------------------------------------- MMA issuer
      const uint32_t p1_own = smem_u32(p1done), p1_peer = map_peer(p1_own, 1);
      const uint32_t p2_own = smem_u32(p2done), p2_peer = map_peer(p2_own, 1);
      bool any = false;
      if (mbar_wait_cluster(ready1, 0, abort_flag)) {
        tc_fence_after();
        mma_tiles(tmem_base, tA, tA, IDESC);  // acc0 = Q Q^T
        any = true;
        umma_commit_pair(p1_own);
        umma_commit_pair(p1_peer);
        if (mbar_wait_cluster(ready2, 0, abort_flag)) {
          tc_fence_after();
          mma_tiles(tmem_base + 256, tB, tA, IDESC);  // acc1 = Q2 W^T
          umma_commit_pair(p2_own);
          umma_commit_pair(p2_peer);
        } else {
          record_timeout(a.status, abort_flag);
        }
      } else {
        record_timeout(a.status, abort_flag);
      }
      if (*abort_flag && any) {  // the MMAs in flight finish before TMEM is released
        umma_commit_pair(smem_u32(drain));
        const unsigned long long t0 = global_timer_ns();
        while (!mbar_try_wait(drain, 0) && global_timer_ns() - t0 < 10000000ull) {
        }
      }
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogues
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;  // which half of the columns
    const int row = quarter * 32 + lane;  // this thread's row (and TMEM lane)
    const int i = 128 * rank + row;       // in the superblock
    const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    bool ok = mbar_wait_cluster(p1done, 0, abort_flag);
    if (!__all_sync(0xffffffffu, ok)) {
      record_timeout(a.status, abort_flag);
    } else {
      tc_fence_after();
      // (1) Q2 = -acc0, W = Q2 - 2Q (bf16 operands); acc0 <- I + 2Q + 2 Q2
#pragma unroll 1
      for (int c0 = 128 * half; c0 < 128 * half + 128; c0 += 32) {
        uint32_t r[32];
        tmem_load_32cols(t_row + c0, r);
        tmem_load_wait();
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int c = c0 + 8 * g;
          const uint32_t off = op_off(row, c);
          const uint4 hv = *reinterpret_cast<const uint4*>(tA + off);
          const uint4 lv = *reinterpret_cast<const uint4*>(tC + off);
          const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
          const uint32_t lw[4] = {lv.x, lv.y, lv.z, lv.w};
          uint32_t w_out[4], q2_out[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float q_a = bf_lo(hw[e]) + bf_lo(lw[e]);
            const float q_b = bf_hi(hw[e]) + bf_hi(lw[e]);
            const float q2_a = -__uint_as_float(r[8 * g + 2 * e]);
            const float q2_b = -__uint_as_float(r[8 * g + 2 * e + 1]);
            __nv_bfloat162 w2 = __floats2bfloat162_rn(q2_a - 2.f * q_a, q2_b - 2.f * q_b);
            __nv_bfloat162 s2 = __floats2bfloat162_rn(q2_a, q2_b);
            w_out[e] = *reinterpret_cast<uint32_t*>(&w2);
            q2_out[e] = *reinterpret_cast<uint32_t*>(&s2);
            const int ca = c + 2 * e;
            r[8 * g + 2 * e] =
                __float_as_uint((i == ca ? 1.f : 0.f) + 2.f * q_a + 2.f * q2_a);
            r[8 * g + 2 * e + 1] =
                __float_as_uint((i == ca + 1 ? 1.f : 0.f) + 2.f * q_b + 2.f * q2_b);
          }
          st_shared_v4(tA + off, w_out[0], w_out[1], w_out[2], w_out[3]);
          st_shared_v4(tB + off, q2_out[0], q2_out[1], q2_out[2], q2_out[3]);
        }
        tmem_store_32cols(t_row + c0, r);
      }
      tmem_store_wait();
      fence_proxy_async_shared();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(map_peer(smem_u32(ready2), 0));
      // (2) the block rows: acc0 + acc1 on the diagonal b-block of row i
      ok = mbar_wait_cluster(p2done, 0, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        record_timeout(a.status, abort_flag);
      } else {
        tc_fence_after();
        const int bl = i / b, ib = i - bl * b;
        uint4* out = reinterpret_cast<uint4*>(
            a.blocks + ((static_cast<long long>(sb) * a.nb + bl) * b + ib) * b);
        // the warp's 32 rows lie in one block (b >= 32): same columns for all
        // lanes; the two warps of a quarter take halves of them (b = 32: one)
        const int cw = b >= 64 ? b / 2 : (half == 0 ? b : 0);
        const int cb = bl * b + (b >= 64 ? half * (b / 2) : 0);
#pragma unroll 1
        for (int c0 = cb; c0 < cb + cw; c0 += 32) {
          uint32_t z[32], y[32];
          tmem_load_32cols(t_row + c0, z);
          tmem_load_32cols(t_row + 256 + c0, y);
          tmem_load_wait();
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            __nv_bfloat162 p2 = __floats2bfloat162_rn(
                __uint_as_float(z[2 * e]) + __uint_as_float(y[2 * e]),
                __uint_as_float(z[2 * e + 1]) + __uint_as_float(y[2 * e + 1]));
            w[e] = *reinterpret_cast<uint32_t*>(&p2);
          }
          uint4* dst = out + (c0 - bl * b) / 8;
#pragma unroll
          for (int q = 0; q < 4; ++q) dst[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still signal or read it
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 512);
  }
}

}  // namespace

bool cnp_pair_fits(int b, int k) { return k == 3 && b >= 32 && b <= 256 && 256 % b == 0; }

cudaError_t cnp_build_pair(const float* theta, int n, int b, __nv_bfloat16* blocks,
                           cudaStream_t stream) {
  if (!cnp_pair_fits(b, 3) || n <= 0 || (static_cast<long long>(n) * b) % 256 != 0)
    return cudaErrorInvalidValue;
  static bool attr_set[64] = {false};
  static std::mutex mu;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_set[dev]) {
      cudaError_t e = cudaFuncSetAttribute(cnp_build_pair_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, kBuildSmem);
      if (e != cudaSuccess) return e;
      attr_set[dev] = true;
    }
  }
  CnpBuildArgs a;
  a.theta = theta;
  a.b = b;
  a.nb = 256 / b;
  a.blocks = blocks;
  a.status = device_status_ptr();
  const long long nsb = static_cast<long long>(n) * b / 256;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * nsb));
  cfg.blockDim = dim3(kCnpThreads);
  cfg.dynamicSmemBytes = kBuildSmem;
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
  prof_begin("cnp_build", stream);
  cudaError_t e = cudaLaunchKernelEx(&cfg, cnp_build_pair_kernel, a);
  prof_end("cnp_build", stream);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace poetx
