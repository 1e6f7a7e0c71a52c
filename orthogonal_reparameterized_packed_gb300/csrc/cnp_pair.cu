// The Cayley-Neumann block build and its adjoint on CTA pairs, every operand
// in shared memory: the pages' fused CNP kernel that loads Q (and Q^2) into
// shared memory once, laid out for two SMs.  k = 3 has kernels of its own
// (two and three dependent phases); any other k >= 1 runs a Horner
// recursion of k phases (further below).
//
// One cluster of two CTAs per 256 x 256 superblock (one block of b = 256, or
// 256 / b blocks of b = 32, 64, 128 on its diagonal: products of block-
// diagonal matrices stay block diagonal).  CTA rank r owns rows 128 r ..
// 128 r + 127 of every matrix; a pair MMA (M = 256 over both CTAs, N = 256,
// D = A B^T) reads A from each CTA's own rows and B from each CTA's own
// rows of the second operand, so with Q^T = -Q and (Q^2)^T = Q^2 the builds
// never transpose or exchange a matrix (the adjoints exchange one MN-major
// tile per phase through distributed shared memory).  The k = 3 build:
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

// ------------------------------------------------ Q from the packed parameters
// The packed rows a CTA reads: b = 256: rank 0 the triangle's rows 0..127,
// rank 1 its rows 128..254 (each a contiguous range); b <= 128: the whole
// triangles of the blocks in this CTA's half.  Bulk copies bring them into
// shared memory (a staging area of at least 98048 bytes).
struct QStage {
  int b, P, lb, bl0, nbl, row0, row1, s0, per_block;
};

__device__ __forceinline__ int tri_start_of(int ib, int b) { return ib * b - ib * (ib + 1) / 2; }

__device__ __forceinline__ QStage qstage_geom(int b, int nb, int rank) {
  QStage q;
  q.b = b;
  q.P = b * (b - 1) / 2;
  q.lb = __ffs(b) - 1;  // b is a power of two
  q.bl0 = b <= 128 ? rank * (nb / 2) : 0;
  q.nbl = b <= 128 ? nb / 2 : 1;
  q.row0 = b <= 128 ? 0 : 128 * rank;           // first staged triangle row
  q.row1 = b <= 128 ? b - 1 : 128 * rank + 128;  // one past the last
  q.s0 = tri_start_of(q.row0, b);
  q.per_block = (q.row1 >= b - 1 ? q.P : tri_start_of(q.row1, b)) - q.s0;
  return q;
}

// One thread: the bulk copies of this CTA's packed rows; `theta_sb` is the
// superblock's first block.
__device__ __forceinline__ void qstage_issue(const QStage& q, const float* theta_sb,
                                             uint8_t* staging, uint64_t* bar) {
  const float* src = theta_sb + static_cast<long long>(q.bl0) * q.P + q.s0;
  const uint32_t bytes = static_cast<uint32_t>(q.nbl * q.per_block) * 4u;
  mbar_arrive_expect_tx(bar, bytes);
  // 16-byte aligned: P * 4 and tri_start(128) * 4 (256-blocks) are multiples of 16
  for (uint32_t off = 0; off < bytes; off += 32768u)
    bulk_load_1d(staging + off, reinterpret_cast<const uint8_t*>(src) + off,
                 bytes - off < 32768u ? bytes - off : 32768u, bar);
}

// All threads of both CTAs: Q of this CTA's rows as bf16 hi (tA) and, if tC
// is given, lo parts.  Every 8-column group of the tiles is written once:
// Q[p][c] = +theta(p, c) (c > p: staged row p), -theta(c, p) (c < p: staged
// row c), 0 on the diagonal and outside the diagonal b-blocks.  For b = 256
// the columns 0..127 of rank 1's rows come from rows 0..127 of the
// triangle, which rank 0 staged: rank 1 reads those from rank 0's shared
// memory.  Items run rows fastest, so a warp covers 32 rows of one group:
// the same branch for almost every lane, and the lower-triangle reads of
// consecutive rows are consecutive words.
__device__ void q_gather(const QStage& q, int rank, const uint8_t* staging, uint64_t* bar,
                         uint8_t* tA, uint8_t* tC, volatile int* abort_flag, int* status) {
  const int b = q.b, lb = q.lb;
  const bool got = mbar_wait(bar, 0, abort_flag);
  if (!got) record_timeout(status, abort_flag);
  if (b == 256) cluster_sync();  // rank 0's staging has landed before rank 1 reads it
  const float* st = reinterpret_cast<const float*>(staging);
  const uint32_t peer_st = map_peer(smem_u32(staging), 0);  // rank 0's staging (b = 256)
  const int lg = lb - 3;  // log2 of the 8-column groups per block row
  if (b <= 128) {  // zeros outside the blocks: 32 - b/8 groups of each row
    const int zg = 32 - (b >> 3);
    for (int t = threadIdx.x; got && t < 128 * zg; t += blockDim.x) {
      const int row = t & 127, k = t >> 7;
      const int p = 128 * rank + row;
      const int own0 = (p >> lb) << lg;  // first group of the row's block
      const int g = k < own0 ? k : k + (b >> 3);
      const uint32_t off = op_off(row, 8 * g);
      st_shared_v4(tA + off, 0u, 0u, 0u, 0u);
      if (tC != nullptr) st_shared_v4(tC + off, 0u, 0u, 0u, 0u);
    }
  }
  const int groups = b <= 128 ? (b >> 3) : 32;  // in-block groups per row
  for (int t = threadIdx.x; got && t < 128 * groups; t += blockDim.x) {
    const int row = t & 127;
    const int p = 128 * rank + row;
    const int blk = p >> lb;
    const int c8 = (blk << lb) + 8 * (t >> 7);
    const int pb = p - (blk << lb), cb = c8 - (blk << lb);  // in-block row, first column
    const float* sblk = st + (blk - q.bl0) * q.per_block - q.s0;  // + tri_start(row) + ...
    float v[8];
    if (cb > pb) {  // upper: row pb of the triangle, entries cb - pb - 1 ..
      const float* r = sblk + tri_start_of(pb, b) + (cb - pb - 1);
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = r[e];
    } else if (cb + 7 < pb) {  // lower: -theta(c, p) from rows c = cb .. cb + 7
      int at = tri_start_of(cb, b) + (pb - cb - 1);
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
        v[e] = c > pb ? sblk[tri_start_of(pb, b) + (c - pb - 1)]
                      : (c < pb ? -sblk[tri_start_of(c, b) + (pb - c - 1)] : 0.f);
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
    if (tC != nullptr) st_shared_v4(tC + off, lw[0], lw[1], lw[2], lw[3]);
  }
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
  const QStage qs = qstage_geom(b, a.nb, rank);
  if (threadIdx.x == 0)
    qstage_issue(qs, a.theta + static_cast<long long>(sb) * a.nb * qs.P, tB, staged);
  q_gather(qs, rank, tB, staged, tA, tC, abort_flag, a.status);
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


// ----------------------------------------------------------- the adjoint
// Gradient of the k = 3 build with respect to the packed parameters, from
// the token sums H = G^T of the block gradient G (split-K partials over
// 256 x 256 superblocks).  With Q^T = -Q, Q2 = Q Q (symmetric) and
// MMA(A, B) = A B^T on own-row tiles (MMA_mn: B read as [K][N]):
//
//   G2  = 2G + G (Q2 - 2Q) + Q2 G            (gradient with respect to Q2)
//   G_Q = 2G + 2 Q2 G - G2 Q - Q G2          (with respect to Q)
//   dtheta[idx(i, j)] = G_Q[i][j] - G_Q[j][i],  i < j
//
//   phase 1   Q (bf16) from theta as in the build; acc0 = MMA(Q, Q) = -Q2;
//             epilogue: Q2, X = 2Q + Q2 (bf16 tiles; X^T = Q2 - 2Q).  This
//             needs theta only and runs before the wait for the partials.
//   sums      H, summed over the K splits into bf16 scratch, by a kernel
//             of its own on all SMs (cnp_sum_partials_kernel) before this
//             one passes its wait
//   phase 2   acc1 = MMA(Q2, H) = Q2 G, acc0 = MMA(G, X) = G (Q2 - 2Q);
//             H's row chunks (B) and G's (A, read MN-major from H's columns:
//             G = H^T is never formed) stream through a two-slot ring of
//             16 KiB chunks (five 64 KiB tiles would not fit)
//   epilogue  G2 = 2G + acc0 + acc1 -> bf16 tile (own rows) and -G2 as an
//             MN-major tile (rows k, this CTA's columns: the other half of
//             each of our rows goes to the peer through distributed shared
//             memory); acc1 <- 2G + 2 acc1
//   phase 3   acc1 += MMA(G2, Q) + MMA_mn(Q, -G2) = ... - G2 Q - Q G2
//   epilogue  G_Q -> fp32 rows in shared memory (rows padded to 257 words;
//             for a 256-block rank 1 sends its columns 0..127 to rank 0,
//             transposed); after a cluster barrier each CTA takes dtheta =
//             G_Q - G_Q^T over the triangle rows it holds, from its own
//             shared memory
//
// Blocks narrower than 256 sit on the superblock's diagonal; the diagonal
// blocks of G_Q depend only on those of G (Q is block diagonal), and the
// sums write H (hence G) as zero outside them.
constexpr int kAdjSlot = BM * BK * 2;  // 16 KiB: a 128 x 64 chunk of G or H
constexpr int kGqPitch = 257;          // words per staged G_Q row (conflict-free columns)
constexpr int kGqOwnBytes = BM * kGqPitch * 4;
static_assert(kGqOwnBytes % 16 == 0 && kGqOwnBytes + BM * 128 * 4 <= 3 * kOpBytes + 2 * kAdjSlot,
              "staged G_Q rows and the transposed quadrant below the barriers");
constexpr int kAdjSmem = 1024 + 3 * kOpBytes + 2 * kAdjSlot + 256;
static_assert(kAdjSmem <= 227 * 1024, "shared memory per CTA");
static_assert(2 * kOpBytes >= (32640 - 8128) * 4, "theta staging in the Q2 and X tiles");

// Byte offset of element (k, n) of an MN-major B tile (K = 256 rows, this
// CTA's 128 columns): per 64-row K step two 64-column chunks of 64 rows x
// 128 bytes, 16-byte groups swizzled with k % 8.
__device__ __forceinline__ uint32_t mn_off(int k, int n) {
  return static_cast<uint32_t>((k >> 6) * 16384 + (n >> 6) * 8192 + (k & 63) * 128 +
                               ((((n & 63) >> 3) ^ (k & 7)) << 4) + ((n & 7) << 1));
}

// One thread, 32 consecutive columns c0.. of its row of G_Q (fp32 bits):
// into its own staged row, or (rank 1 of a 256-block, columns < 128) into
// rank 0's transposed quadrant at [c][row] (cross: that quadrant's shared::
// cluster address plus 4 * row).
__device__ __forceinline__ void stage_gq32(const uint32_t (&r)[32], int c0, bool to_peer,
                                           float* own_row, uint32_t cross) {
  if (to_peer) {
#pragma unroll
    for (int e = 0; e < 32; ++e) st_cluster_b32(cross + 4u * static_cast<uint32_t>((c0 + e) * 128), r[e]);
  } else {
#pragma unroll
    for (int e = 0; e < 32; ++e) own_row[c0 + e] = __uint_as_float(r[e]);
  }
}

// All threads of a CTA, after both CTAs staged G_Q: dtheta = G_Q - G_Q^T
// over the upper triangles of the blocks whose rows this CTA holds, from
// shared memory only.  b <= 128: whole blocks; b = 256: rank 0 takes the
// triangle's rows 0..127 (the quadrant of rows 128.. it reads transposed
// from gq_cross), rank 1 rows 128..254.
__device__ void pack_dtheta(int b, int lb, int P, int rank, int lsb, int nb, float* dtheta,
                            const float* gq_own, const float* gq_cross) {
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t own_s = smem_u32(gq_own), cross_s = smem_u32(gq_cross);
  const int bpc = b <= 128 ? 128 / b : 1;               // blocks per CTA
  const int rows_per = b <= 128 ? b - 1 : 128 - rank;  // triangle rows per block here
  for (int r = warp; r < bpc * rows_per; r += blockDim.x / 32) {
    const int blo = r / rows_per, rr = r - blo * rows_per;
    const int il = b <= 128 ? blo * b + rr : rr;  // local row
    const int i = 128 * rank + il;                // superblock row
    const int ib = i & (b - 1);                   // row in its block
    const int cb0 = i - ib;                       // the block's first column
    const int bl = cb0 >> lb;
    float* dst = dtheta + (static_cast<long long>(lsb) * nb + bl) * P + tri_start_of(ib, b) - ib - 1;
    const uint32_t rowi = own_s + 4u * static_cast<uint32_t>(il * kGqPitch + cb0);
    for (int j0 = ib + 1 + lane; j0 < b; j0 += 128) {
      float d4[4];  // four columns' loads before the stores
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int jb = min(j0 + 32 * u, b - 1);
        const int j = cb0 + jb;  // superblock column = row of the transposed entry
        const uint32_t at_ji = j - 128 * rank < 128
                                   ? own_s + 4u * static_cast<uint32_t>((j - 128 * rank) * kGqPitch + i)
                                   : cross_s + 4u * static_cast<uint32_t>(i * 128 + (j - 128));
        d4[u] = ld_shared_f32(rowi + 4u * static_cast<uint32_t>(jb)) - ld_shared_f32(at_ji);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (j0 + 32 * u < b) dst[j0 + 32 * u] = d4[u];
    }
  }
}

struct CnpAdjArgs;
__global__ void cnp_sum_partials_kernel(const CnpAdjArgs a);

struct CnpAdjArgs {
  const float* theta_a;
  const float* theta_b;
  const float* part_a;  // [splits_a][nsb_a][256][256] fp32, = H
  const float* part_b;
  int splits_a, splits_b, nsb_a, nsb_b;
  int b, nb;
  __nv_bfloat16* hg;  // [nsb_a + nsb_b][256][256] bf16 scratch: H
  float* dtheta_a;
  float* dtheta_b;
  int* status;
};

// The token sums H of every superblock of both sides: the split-K
// partials [splits][superblocks][256][256] (fp32) summed, rounded to bf16
// into hg (zero outside the diagonal b-blocks).  One 8-column group of a
// row per thread, four splits' loads in flight; all SMs, ahead of the
// adjoint.  It lets the adjoint launch before it waits itself: the adjoint
// reads only theta before its own wait (no kernel that may still run writes
// theta: the kernels before this one's predecessor are complete once that
// predecessor has been launched), and after its wait this kernel is done.
__global__ void __launch_bounds__(256) cnp_sum_partials_kernel(const CnpAdjArgs a) {
  pdl_trigger();
  pdl_wait();  // the partials are complete from here on
  const int lb = __ffs(a.b) - 1;
  const long long items = static_cast<long long>(a.nsb_a + a.nsb_b) * 256 * 32;
  for (long long it = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; it < items;
       it += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int sb = static_cast<int>(it >> 13);  // 8192 groups per superblock
    const int p = static_cast<int>(it >> 5) & 255;
    const int c8 = 8 * static_cast<int>(it & 31);
    const bool side_b = sb >= a.nsb_a;
    const int lsb = side_b ? sb - a.nsb_a : sb;
    const long long split_stride = static_cast<long long>(side_b ? a.nsb_b : a.nsb_a) * 65536;
    const int splits = side_b ? a.splits_b : a.splits_a;
    const float* ps = (side_b ? a.part_b : a.part_a) + static_cast<long long>(lsb) * 65536 + p * 256 + c8;
    float h[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) h[e] = 0.f;
    if ((c8 >> lb) == (p >> lb)) {
      int sp = 0;
      for (; sp + 4 <= splits; sp += 4) {
        float4 v[8];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          v[2 * u] = *reinterpret_cast<const float4*>(ps + (sp + u) * split_stride);
          v[2 * u + 1] = *reinterpret_cast<const float4*>(ps + (sp + u) * split_stride + 4);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          h[0] += v[2 * u].x; h[1] += v[2 * u].y; h[2] += v[2 * u].z; h[3] += v[2 * u].w;
          h[4] += v[2 * u + 1].x; h[5] += v[2 * u + 1].y; h[6] += v[2 * u + 1].z;
          h[7] += v[2 * u + 1].w;
        }
      }
      for (; sp < splits; ++sp) {
        const float4 v0 = *reinterpret_cast<const float4*>(ps + sp * split_stride);
        const float4 v1 = *reinterpret_cast<const float4*>(ps + sp * split_stride + 4);
        h[0] += v0.x; h[1] += v0.y; h[2] += v0.z; h[3] += v0.w;
        h[4] += v1.x; h[5] += v1.y; h[6] += v1.z; h[7] += v1.w;
      }
    }
    uint32_t hw[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat162 hh = __floats2bfloat162_rn(h[2 * e], h[2 * e + 1]);
      hw[e] = *reinterpret_cast<const uint32_t*>(&hh);
    }
    *reinterpret_cast<uint4*>(a.hg + (static_cast<long long>(sb) * 256 + p) * 256 + c8) =
        make_uint4(hw[0], hw[1], hw[2], hw[3]);
  }
}

__global__ void __launch_bounds__(kCnpThreads, 1)
    cnp_adjoint_pair_kernel(const __grid_constant__ CUtensorMap tmH,
                            const __grid_constant__ CUtensorMap tmHmn, const CnpAdjArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* tQ = base;                  // Q (bf16 hi)
  uint8_t* tQ2 = base + kOpBytes;      // theta staging; Q2; then G2
  uint8_t* tX = base + 2 * kOpBytes;   // (staging); X; then -G2 as an MN-major tile
  uint8_t* slots = base + 3 * kOpBytes;
  // after phase 3: G_Q rows of this CTA (pitch kGqPitch) and, in rank 0 of a
  // 256-block, the transposed quadrant G_Q[128 + jj][c] at [c][jj]
  float* gq_own = reinterpret_cast<float*>(base);
  float* gq_cross = reinterpret_cast<float*>(base + kGqOwnBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(slots + 2 * kAdjSlot);
  uint64_t* ready1 = bars + 0;   // leader: Q tiles written (one arrival per CTA)
  uint64_t* p1done = bars + 1;   // each CTA
  uint64_t* ready2 = bars + 2;   // leader: Q2, X written (eight warps per CTA)
  uint64_t* full = bars + 3;     // [2] leader: a chunk pair has landed
  uint64_t* empty = bars + 5;    // [2] each CTA: the slot is free
  uint64_t* p2done = bars + 7;   // each CTA
  uint64_t* ready3 = bars + 8;   // leader: G2 tiles written (eight warps per CTA)
  uint64_t* p3done = bars + 9;   // each CTA
  uint64_t* drain = bars + 10;
  uint64_t* staged = bars + 11;  // the theta bulk copy has landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 12);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int rank = static_cast<int>(cluster_ctarank());
  const bool leader = rank == 0;
  const bool issuer = warp == 1 && lane == 0 && leader;
  const int sb = static_cast<int>(cluster_id_x());  // superblock over both sides
  const bool side_b = sb >= a.nsb_a;
  const int lsb = side_b ? sb - a.nsb_a : sb;
  const float* theta = side_b ? a.theta_b : a.theta_a;
  float* dtheta = side_b ? a.dtheta_b : a.dtheta_a;
  const int b = a.b;
  const int lb = __ffs(b) - 1;

  if (threadIdx.x == 0) {
    mbar_init(ready1, 2);
    mbar_init(p1done, 1);
    mbar_init(ready2, 16);
    for (int q = 0; q < 2; ++q) {
      mbar_init(&full[q], 1);
      mbar_init(&empty[q], 1);
    }
    mbar_init(p2done, 1);
    mbar_init(ready3, 16);
    mbar_init(p3done, 1);
    mbar_init(drain, 1);
    mbar_init(staged, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmH);
    tma_prefetch_desc(&tmHmn);
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

  // ---------------------------------------------- from theta alone (phase 1)
  // theta is no kernel's output in this stream's recent past (every kernel
  // here waits for its predecessor before it lets a successor start), so
  // this part may overlap the end of the kernel that writes the partials.
  const QStage qs = qstage_geom(b, a.nb, rank);
  if (threadIdx.x == 0)
    qstage_issue(qs, theta + static_cast<long long>(lsb) * a.nb * qs.P, tQ2, staged);
  q_gather(qs, rank, tQ2, staged, tQ, nullptr, abort_flag, a.status);
  fence_proxy_async_all();
  cluster_sync();  // Q tiles complete in both CTAs
  if (threadIdx.x == 0) mbar_arrive_remote(map_peer(smem_u32(ready1), 0));

  constexpr uint32_t IDESC = instr_desc_bf16(2 * BM, 256, false, false);
  constexpr uint32_t IDESC_MN = instr_desc_bf16(2 * BM, 256, false, true);
  constexpr uint32_t IDESC_AMN = instr_desc_bf16(2 * BM, 256, true, false);
  bool mma_ok = true, mma_any = false;  // the issuer's state
  if (issuer) {
    mma_ok = mbar_wait_cluster(ready1, 0, abort_flag);
    if (mma_ok) {
      tc_fence_after();
      mma_tiles(tmem_base, tQ, tQ, IDESC);  // acc0 = Q Q^T = -Q2
      mma_any = true;
      umma_commit_pair(smem_u32(p1done));
      umma_commit_pair(map_peer(smem_u32(p1done), 1));
    }
  }
  // epilogue warps: four row quarters x two column halves
  const int quarter = warp & 3;
  const int half = (warp - 2) >> 2;
  const int row = quarter * 32 + lane;
  const int p = 128 * rank + row;  // in the superblock
  const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
  bool epi_ok = true;
  if (warp >= 2) {
    // (1) Q2 = -acc0 and X = 2Q + Q2 (bf16 tiles, own rows)
    epi_ok = __all_sync(0xffffffffu, mbar_wait_cluster(p1done, 0, abort_flag));
    if (epi_ok) {
      tc_fence_after();
#pragma unroll 1
      for (int c0 = 128 * half; c0 < 128 * half + 128; c0 += 32) {
        uint32_t r[32];
        tmem_load_32cols(t_row + c0, r);
        tmem_load_wait();
#pragma unroll
        for (int gi = 0; gi < 4; ++gi) {
          const uint32_t off = op_off(row, c0 + 8 * gi);
          const uint4 qv = *reinterpret_cast<const uint4*>(tQ + off);
          const uint32_t qw[4] = {qv.x, qv.y, qv.z, qv.w};
          uint32_t q2w[4], xw[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float q2a = -__uint_as_float(r[8 * gi + 2 * e]);
            const float q2b = -__uint_as_float(r[8 * gi + 2 * e + 1]);
            const __nv_bfloat162 s2 = __floats2bfloat162_rn(q2a, q2b);
            const __nv_bfloat162 x2 =
                __floats2bfloat162_rn(2.f * bf_lo(qw[e]) + q2a, 2.f * bf_hi(qw[e]) + q2b);
            q2w[e] = *reinterpret_cast<const uint32_t*>(&s2);
            xw[e] = *reinterpret_cast<const uint32_t*>(&x2);
          }
          st_shared_v4(tQ2 + off, q2w[0], q2w[1], q2w[2], q2w[3]);
          st_shared_v4(tX + off, xw[0], xw[1], xw[2], xw[3]);
        }
      }
      fence_proxy_async_shared();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(map_peer(smem_u32(ready2), 0));
    } else {
      record_timeout(a.status, abort_flag);
    }
  }

  // ---------------------------------------------- the token sums H (ready)
  pdl_wait();  // the sums kernel is complete: H is in the scratch
  pdl_trigger();
  __syncthreads();
  cluster_sync();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ producer (both CTAs)
      // chunks 0..3: H's rows (B of MMA(Q2, H), K-major); 4..7: G's rows as
      // an MN-major A (64 rows k of H, this CTA's 128 columns, two boxes)
      const uint32_t full0 = map_peer(smem_u32(full), 0);
      const int hrow = sb * 256 + 128 * rank;
      bool ok = true;
      for (int q = 0; q < 8 && ok; ++q) {
        const int slot = q & 1;
        const uint32_t ph = static_cast<uint32_t>(q >> 1) & 1u;
        if (!mbar_wait_cluster(&empty[slot], ph ^ 1, abort_flag)) {
          record_timeout(a.status, abort_flag);
          ok = false;
          break;
        }
        if (leader) mbar_arrive_expect_tx(&full[slot], 2 * kAdjSlot);
        const uint32_t bar = full0 + static_cast<uint32_t>(slot * 8);
        uint8_t* dst = slots + slot * kAdjSlot;
        if (q < 4) {
          tma_load_2d_pair(dst, &tmH, bar, (q & 3) * BK, hrow);
        } else {
          const int krow = sb * 256 + (q & 3) * BK;
          tma_load_2d_pair(dst, &tmHmn, bar, 128 * rank, krow);
          tma_load_2d_pair(dst + 8192, &tmHmn, bar, 128 * rank + 64, krow);
        }
      }
      // the last two chunks are released before the CTA may leave (bounded)
      for (int q = 6; q < 8 && ok; ++q) {
        const unsigned long long t0 = global_timer_ns();
        while (!mbar_try_wait_cluster(&empty[q & 1], static_cast<uint32_t>(q >> 1) & 1u) &&
               global_timer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else if (warp == 1) {
    if (issuer) {
      // ----------------------------------------------------------- MMA issuer
      const uint32_t p2_own = smem_u32(p2done), p2_peer = map_peer(p2_own, 1);
      const uint32_t p3_own = smem_u32(p3done), p3_peer = map_peer(p3_own, 1);
      const uint32_t e_own = smem_u32(empty), e_peer = map_peer(e_own, 1);
      bool ok = mma_ok && mbar_wait_cluster(ready2, 0, abort_flag);
      // acc1 = Q2 H^T (= Q2 G), acc0 = G X^T (= G (Q2 - 2Q))
      for (int q = 0; q < 8 && ok; ++q) {
        const int slot = q & 1, kc = q & 3;
        if (!mbar_wait_cluster(&full[slot], static_cast<uint32_t>(q >> 1) & 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ch = smem_u32(slots + slot * kAdjSlot);
#pragma unroll
        for (int j = 0; j < BK / 16; ++j) {
          const uint32_t acc = (kc > 0 || j > 0) ? 1u : 0u;
          if (q < 4) {
            const uint64_t adesc = smem_desc_sw128(smem_u32(tQ2) + kc * (BM * 128) + j * 32, 16, 1024);
            umma_bf16_pair(tmem_base + 256, adesc, smem_desc_sw128(ch + j * 32, 16, 1024), IDESC, acc);
          } else {  // G read MN-major: its rows are H's columns
            const uint64_t adesc = smem_desc_sw128(ch + j * 2048, 8192, 1024);
            const uint64_t bdesc = smem_desc_sw128(smem_u32(tX) + kc * (BM * 128) + j * 32, 16, 1024);
            umma_bf16_pair(tmem_base, adesc, bdesc, IDESC_AMN, acc);
          }
        }
        umma_commit_pair(e_own + static_cast<uint32_t>(slot * 8));
        umma_commit_pair(e_peer + static_cast<uint32_t>(slot * 8));
      }
      if (ok) {
        umma_commit_pair(p2_own);
        umma_commit_pair(p2_peer);
        ok = mbar_wait_cluster(ready3, 0, abort_flag);
      }
      if (ok) {
        tc_fence_after();
        // acc1 += G2 Q^T (= -G2 Q) + Q (-G2)
        const uint32_t g2 = smem_u32(tQ2), q0 = smem_u32(tQ), mn = smem_u32(tX);
#pragma unroll
        for (int kc = 0; kc < 4; ++kc)
#pragma unroll
          for (int j = 0; j < BK / 16; ++j) {
            umma_bf16_pair(tmem_base + 256,
                           smem_desc_sw128(g2 + kc * (BM * 128) + j * 32, 16, 1024),
                           smem_desc_sw128(q0 + kc * (BM * 128) + j * 32, 16, 1024), IDESC, 1u);
            umma_bf16_pair(tmem_base + 256,
                           smem_desc_sw128(q0 + kc * (BM * 128) + j * 32, 16, 1024),
                           smem_desc_sw128(mn + kc * 16384 + j * 2048, 8192, 1024), IDESC_MN, 1u);
          }
        umma_commit_pair(p3_own);
        umma_commit_pair(p3_peer);
      }
      if (!ok) record_timeout(a.status, abort_flag);
      if (!ok && mma_any) {  // the MMAs in flight finish before TMEM is released
        umma_commit_pair(smem_u32(drain));
        const unsigned long long t0 = global_timer_ns();
        while (!mbar_try_wait(drain, 0) && global_timer_ns() - t0 < 10000000ull) {
        }
      }
    }
  } else if (epi_ok) {
    // ------------------------------------------------------------ epilogues
    const uint32_t mnX[2] = {map_peer(smem_u32(tX), 0), map_peer(smem_u32(tX), 1)};
    // G[p][c] = H[c][p]: for a fixed c the warp's 32 rows are consecutive
    // elements of H's row c (written by either CTA); the first 32 columns
    // are fetched while phase 2 runs
    const __nv_bfloat16* hcol = a.hg + static_cast<long long>(sb) * 65536 + p;
    float gcol[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) gcol[e] = __bfloat162float(hcol[(128 * half + e) * 256]);
    // (2) G2 = 2G + acc0 + acc1: own-row tile and -G2 as MN tiles;
    //     acc1 <- 2G + 2 acc1
    bool ok = __all_sync(0xffffffffu, mbar_wait_cluster(p2done, 0, abort_flag));
    if (ok) {
      tc_fence_after();
#pragma unroll 1
      for (int c0 = 128 * half; c0 < 128 * half + 128; c0 += 32) {
        uint32_t r[32], s[32];
        tmem_load_32cols(t_row + c0, r);
        tmem_load_32cols(t_row + 256 + c0, s);
        tmem_load_wait();
#pragma unroll
        for (int gi = 0; gi < 4; ++gi) {
          uint32_t pw[4], nw[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int ia = 8 * gi + 2 * e;
            const float ga = gcol[ia], gb = gcol[ia + 1];
            const float sa = __uint_as_float(s[ia]), sv = __uint_as_float(s[ia + 1]);
            const float g2a = 2.f * ga + __uint_as_float(r[ia]) + sa;
            const float g2b = 2.f * gb + __uint_as_float(r[ia + 1]) + sv;
            const __nv_bfloat162 pz = __floats2bfloat162_rn(g2a, g2b);
            const __nv_bfloat162 nz = __floats2bfloat162_rn(-g2a, -g2b);
            pw[e] = *reinterpret_cast<const uint32_t*>(&pz);
            nw[e] = *reinterpret_cast<const uint32_t*>(&nz);
            s[ia] = __float_as_uint(2.f * ga + 2.f * sa);
            s[ia + 1] = __float_as_uint(2.f * gb + 2.f * sv);
          }
          const int c = c0 + 8 * gi;
          st_shared_v4(tQ2 + op_off(row, c), pw[0], pw[1], pw[2], pw[3]);
          // -G2[p][c..c+7] is row k = p, columns c of the MN tile of the
          // CTA that owns columns c (this one or the peer)
          st_cluster_v4(mnX[c >> 7] + mn_off(p, c & 127), nw[0], nw[1], nw[2], nw[3]);
        }
        tmem_store_32cols(t_row + 256 + c0, s);
        if (c0 + 32 < 128 * half + 128) {
#pragma unroll
          for (int e = 0; e < 32; ++e) gcol[e] = __bfloat162float(hcol[(c0 + 32 + e) * 256]);
        }
      }
      tmem_store_wait();
      fence_proxy_async_all();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(map_peer(smem_u32(ready3), 0));
      // (3) G_Q = acc1 -> fp32 rows in shared memory.  Phase 3 has read
      //     every operand tile of both CTAs once p3done completes, and the
      //     peer wrote its last -G2 values into X before phase 3 began.
      //     For a 256-block rank 1's columns 0..127 go to rank 0, transposed.
      ok = __all_sync(0xffffffffu, mbar_wait_cluster(p3done, 0, abort_flag));
      if (ok) {
        tc_fence_after();
        const bool to_peer = b == 256 && rank == 1 && half == 0;
        const uint32_t cross = map_peer(smem_u32(gq_cross), 0) + 4u * static_cast<uint32_t>(row);
        float* own = gq_own + row * kGqPitch;
#pragma unroll 1
        for (int c0 = 128 * half; c0 < 128 * half + 128; c0 += 32) {
          uint32_t r[32];
          tmem_load_32cols(t_row + 256 + c0, r);
          tmem_load_wait();
          stage_gq32(r, c0, to_peer, own, cross);
        }
      } else {
        record_timeout(a.status, abort_flag);
      }
    } else {
      record_timeout(a.status, abort_flag);
    }
  }

  // ------------------------------------------------------------------ pack
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // G_Q staged in both CTAs
  pack_dtheta(b, lb, qs.P, rank, lsb, a.nb, dtheta, gq_own, gq_cross);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still signal or read it
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 512);
  }
}

// ------------------------------------------------- the build for any k >= 1
// E_{k+1} = Q,  E_i = 2Q + E_{i+1} Q  (i = k .. 1),  R = I + E_1, i.e.
// R = I + 2Q + ... + 2Q^k + Q^{k+1}.  With MMA(A, B) = A B^T and Q^T = -Q,
// E_{i+1} Q = -MMA(E_{i+1}, Q): both operands are a CTA's own rows, so the
// k phases exchange nothing:
//   phase i   acc = MMA(E, Q_hi)            (E = Q_hi in the first phase)
//   epilogue  E = 2Q - acc -> bf16 tile      (2Q from the hi and lo parts)
//   last      block rows = I + 2Q - acc -> bf16
// Same shared-memory layout as the k = 3 build (Q hi, Q lo, staging then E).
__global__ void __launch_bounds__(kCnpThreads, 1) cnp_build_pair_k_kernel(const CnpBuildArgs a,
                                                                          int k) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* tA = base;                 // Q hi
  uint8_t* tC = base + kOpBytes;      // Q lo
  uint8_t* tB = base + 2 * kOpBytes;  // staged theta, then E
  uint64_t* ready1 = reinterpret_cast<uint64_t*>(base + 2 * kOpBytes + kStageBytes);
  uint64_t* pdone = ready1 + 1;   // each CTA: a phase's MMAs are done (parity: phase % 2)
  uint64_t* readyE = pdone + 1;   // leader: E written (eight warps of each CTA)
  uint64_t* drain = readyE + 1;
  uint64_t* staged = drain + 1;
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
    mbar_init(pdone, 1);
    mbar_init(readyE, 16);
    mbar_init(drain, 1);
    mbar_init(staged, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, 256);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  pdl_trigger();

  const QStage qs = qstage_geom(b, a.nb, rank);
  if (threadIdx.x == 0)
    qstage_issue(qs, a.theta + static_cast<long long>(sb) * a.nb * qs.P, tB, staged);
  q_gather(qs, rank, tB, staged, tA, tC, abort_flag, a.status);
  fence_proxy_async_all();
  cluster_sync();  // both CTAs' Q tiles are complete; the staging is free
  if (threadIdx.x == 0) mbar_arrive_remote(map_peer(smem_u32(ready1), 0));

  constexpr uint32_t IDESC = instr_desc_bf16(2 * BM, 256, false, false);
  if (warp == 1) {
    if (lane == 0 && leader) {
      // ----------------------------------------------------------- MMA issuer
      const uint32_t pd_own = smem_u32(pdone), pd_peer = map_peer(pd_own, 1);
      bool ok = mbar_wait_cluster(ready1, 0, abort_flag), any = false;
      for (int ph = 0; ph < k && ok; ++ph) {
        if (ph > 0 && !mbar_wait_cluster(readyE, static_cast<uint32_t>(ph - 1) & 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        mma_tiles(tmem_base, ph == 0 ? tA : tB, tA, IDESC);  // acc = E Q^T
        any = true;
        umma_commit_pair(pd_own);
        umma_commit_pair(pd_peer);
      }
      if (!ok) record_timeout(a.status, abort_flag);
      if (!ok && any) {  // the MMAs in flight finish before TMEM is released
        umma_commit_pair(smem_u32(drain));
        const unsigned long long t0 = global_timer_ns();
        while (!mbar_try_wait(drain, 0) && global_timer_ns() - t0 < 10000000ull) {
        }
      }
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogues
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    const int i = 128 * rank + row;
    const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    for (int ph = 0; ph < k; ++ph) {
      const bool ok = mbar_wait_cluster(pdone, static_cast<uint32_t>(ph) & 1u, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        record_timeout(a.status, abort_flag);
        break;
      }
      tc_fence_after();
      if (ph + 1 < k) {
        // E = 2Q - acc over this half's 128 columns, bf16 into the E tile
#pragma unroll 1
        for (int c0 = 128 * half; c0 < 128 * half + 128; c0 += 32) {
          uint32_t r[32];
          tmem_load_32cols(t_row + c0, r);
          tmem_load_wait();
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const uint32_t off = op_off(row, c0 + 8 * g);
            const uint4 hv = *reinterpret_cast<const uint4*>(tA + off);
            const uint4 lv = *reinterpret_cast<const uint4*>(tC + off);
            const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
            const uint32_t lw[4] = {lv.x, lv.y, lv.z, lv.w};
            uint32_t e_out[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float qa = bf_lo(hw[e]) + bf_lo(lw[e]), qb = bf_hi(hw[e]) + bf_hi(lw[e]);
              const __nv_bfloat162 v = __floats2bfloat162_rn(
                  2.f * qa - __uint_as_float(r[8 * g + 2 * e]),
                  2.f * qb - __uint_as_float(r[8 * g + 2 * e + 1]));
              e_out[e] = *reinterpret_cast<const uint32_t*>(&v);
            }
            st_shared_v4(tB + off, e_out[0], e_out[1], e_out[2], e_out[3]);
          }
        }
        fence_proxy_async_shared();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(map_peer(smem_u32(readyE), 0));
      } else {
        // the block rows: I + 2Q - acc on the diagonal b-block of row i
        const int bl = i / b, ib = i - bl * b;
        uint4* out = reinterpret_cast<uint4*>(
            a.blocks + ((static_cast<long long>(sb) * a.nb + bl) * b + ib) * b);
        const int cw = b >= 64 ? b / 2 : (half == 0 ? b : 0);
        const int cb = bl * b + (b >= 64 ? half * (b / 2) : 0);
#pragma unroll 1
        for (int c0 = cb; c0 < cb + cw; c0 += 32) {
          uint32_t r[32];
          tmem_load_32cols(t_row + c0, r);
          tmem_load_wait();
          uint32_t w[16];
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const uint32_t off = op_off(row, c0 + 8 * g);
            const uint4 hv = *reinterpret_cast<const uint4*>(tA + off);
            const uint4 lv = *reinterpret_cast<const uint4*>(tC + off);
            const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w};
            const uint32_t lw[4] = {lv.x, lv.y, lv.z, lv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int ca = c0 + 8 * g + 2 * e;
              const float qa = bf_lo(hw[e]) + bf_lo(lw[e]), qb = bf_hi(hw[e]) + bf_hi(lw[e]);
              const __nv_bfloat162 v = __floats2bfloat162_rn(
                  (i == ca ? 1.f : 0.f) + 2.f * qa - __uint_as_float(r[8 * g + 2 * e]),
                  (i == ca + 1 ? 1.f : 0.f) + 2.f * qb - __uint_as_float(r[8 * g + 2 * e + 1]));
              w[4 * g + e] = *reinterpret_cast<const uint32_t*>(&v);
            }
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
    tmem_dealloc_pair(tmem_base, 256);
  }
}

// ----------------------------------------------- the adjoint for any k >= 1
// With H = G^T (the token sums) and D = (dL/dQ)^T, the reverse sweep of the
// build (Gbar_1 = G, dQ += 2 Gbar_i + E_{i+1}^T Gbar_i, Gbar_{i+1} = Gbar_i Q^T,
// dQ += Gbar_{k+1}) regrouped by Horner's rule on both sides of H:
//   P = H, Y = H;  for m = 0 .. k-1:  P <- 2H + P Q,  Y <- P + Q Y;   D = Y
// (P_m = H a_m(Q) with a_m(x) = 2 + 2x + .. + 2x^m + x^{m+1} = 2I + E_{k-m}
// transposed; Y accumulates Q^p H a_{k-1-p}(Q) + Q^k H).  Both recursions
// run forward, so no E_i is stored.  dtheta(i, j) = dQ[i][j] - dQ[j][i] =
// D[j][i] - D[i][j]: -D is staged and packed like G_Q of the k = 3 adjoint.
//   prologue  Q hi from theta (before the wait for the token sums, which
//             the sums kernel leaves in bf16 scratch); P's tile (H's own
//             rows, K-major) and Y's tile (H read MN-major: rows k, this
//             CTA's columns) by TMA
//   phase m   accP = MMA(P, Q_hi) = -P Q,  accY = MMA_mn(Q_hi, Y) = Q Y
//   epilogue  P = 2H - accP -> bf16 (own rows), Y = P + accY -> bf16 MN tile
//             (the half of each row in the peer's columns through
//             distributed shared memory); in the last phase -Y -> fp32 rows
//             in shared memory, then the pack
// Shared memory as the k = 3 adjoint (Q, then P and Y in the Q2 and X
// places; the staged G_Q rows over all of it).
__global__ void __launch_bounds__(kCnpThreads, 1)
    cnp_adjoint_pair_k_kernel(const __grid_constant__ CUtensorMap tmH,
                              const __grid_constant__ CUtensorMap tmHmn, const CnpAdjArgs a, int k) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* tQ = base;                 // Q hi
  uint8_t* tP = base + kOpBytes;      // theta staging; then P (own rows, K-major)
  uint8_t* tY = base + 2 * kOpBytes;  // (staging); then Y (MN-major, this CTA's columns)
  float* gq_own = reinterpret_cast<float*>(base);
  float* gq_cross = reinterpret_cast<float*>(base + kGqOwnBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + 3 * kOpBytes + 2 * kAdjSlot);
  uint64_t* readyH = bars + 0;   // leader: P and Y tiles of H loaded (one arrival per CTA)
  uint64_t* pdone = bars + 1;    // each CTA; parity: phase % 2
  uint64_t* readyE = bars + 2;   // leader: P and Y written (eight warps per CTA)
  uint64_t* hload = bars + 3;    // each CTA: its TMA loads of H landed
  uint64_t* drain = bars + 4;
  uint64_t* staged = bars + 5;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 6);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int rank = static_cast<int>(cluster_ctarank());
  const bool leader = rank == 0;
  const int sb = static_cast<int>(cluster_id_x());
  const bool side_b = sb >= a.nsb_a;
  const int lsb = side_b ? sb - a.nsb_a : sb;
  const float* theta = side_b ? a.theta_b : a.theta_a;
  float* dtheta = side_b ? a.dtheta_b : a.dtheta_a;
  const int b = a.b;
  const int lb = __ffs(b) - 1;

  if (threadIdx.x == 0) {
    mbar_init(readyH, 2);
    mbar_init(pdone, 1);
    mbar_init(readyE, 16);
    mbar_init(hload, 1);
    mbar_init(drain, 1);
    mbar_init(staged, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmH);
    tma_prefetch_desc(&tmHmn);
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

  // Q from theta alone: may overlap the end of the previous kernel (theta is
  // no recent kernel's output: every kernel here waits before it triggers)
  const QStage qs = qstage_geom(b, a.nb, rank);
  if (threadIdx.x == 0)
    qstage_issue(qs, theta + static_cast<long long>(lsb) * a.nb * qs.P, tP, staged);
  q_gather(qs, rank, tP, staged, tQ, nullptr, abort_flag, a.status);

  pdl_wait();  // the sums kernel is complete: H is in the scratch
  pdl_trigger();
  fence_proxy_async_all();  // the Q tile and the staging reads -> the async proxy
  __syncthreads();
  cluster_sync();  // H and both CTAs' Q tiles complete
  if (threadIdx.x == 0) {
    // P = H's own rows (four 128 x 64 K-major chunks), Y = H MN-major: rows
    // k of the superblock, this CTA's 128 columns (two 64-column boxes per
    // 64-row K step)
    mbar_arrive_expect_tx(hload, 2 * kOpBytes);
    const int hrow = sb * 256 + 128 * rank;
    for (int kc = 0; kc < 4; ++kc) {
      tma_load_2d(tP + kc * (BM * 128), &tmH, hload, kc * BK, hrow);
      tma_load_2d(tY + kc * 16384, &tmHmn, hload, 128 * rank, sb * 256 + kc * BK);
      tma_load_2d(tY + kc * 16384 + 8192, &tmHmn, hload, 128 * rank + 64, sb * 256 + kc * BK);
    }
    if (mbar_wait(hload, 0, abort_flag))
      mbar_arrive_remote(map_peer(smem_u32(readyH), 0));
    else
      record_timeout(a.status, abort_flag);
  }

  constexpr uint32_t IDESC = instr_desc_bf16(2 * BM, 256, false, false);
  constexpr uint32_t IDESC_MN = instr_desc_bf16(2 * BM, 256, false, true);
  if (warp == 1) {
    if (lane == 0 && leader) {
      // ----------------------------------------------------------- MMA issuer
      const uint32_t pd_own = smem_u32(pdone), pd_peer = map_peer(pd_own, 1);
      bool ok = mbar_wait_cluster(readyH, 0, abort_flag), any = false;
      const uint32_t q0 = smem_u32(tQ), y0 = smem_u32(tY);
      for (int m = 0; m < k && ok; ++m) {
        if (m > 0 && !mbar_wait_cluster(readyE, static_cast<uint32_t>(m - 1) & 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        mma_tiles(tmem_base, tP, tQ, IDESC);  // accP = P Q^T = -P Q
#pragma unroll
        for (int kc = 0; kc < 4; ++kc)
#pragma unroll
          for (int j = 0; j < BK / 16; ++j)  // accY = Q Y
            umma_bf16_pair(tmem_base + 256,
                           smem_desc_sw128(q0 + kc * (BM * 128) + j * 32, 16, 1024),
                           smem_desc_sw128(y0 + kc * 16384 + j * 2048, 8192, 1024), IDESC_MN,
                           (kc > 0 || j > 0) ? 1u : 0u);
        any = true;
        umma_commit_pair(pd_own);
        umma_commit_pair(pd_peer);
      }
      if (!ok) record_timeout(a.status, abort_flag);
      if (!ok && any) {
        umma_commit_pair(smem_u32(drain));
        const unsigned long long t0 = global_timer_ns();
        while (!mbar_try_wait(drain, 0) && global_timer_ns() - t0 < 10000000ull) {
        }
      }
    }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ epilogues
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    const int p = 128 * rank + row;
    const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t mnY[2] = {map_peer(smem_u32(tY), 0), map_peer(smem_u32(tY), 1)};
    const uint4* hrow = reinterpret_cast<const uint4*>(a.hg + (static_cast<long long>(sb) * 256 + p) * 256);
    for (int m = 0; m < k; ++m) {
      const bool last = m + 1 == k;
      const bool ok = mbar_wait_cluster(pdone, static_cast<uint32_t>(m) & 1u, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        record_timeout(a.status, abort_flag);
        break;
      }
      tc_fence_after();
      const bool to_peer = last && b == 256 && rank == 1 && half == 0;
      const uint32_t cross = map_peer(smem_u32(gq_cross), 0) + 4u * static_cast<uint32_t>(row);
      float* own = gq_own + row * kGqPitch;
#pragma unroll 1
      for (int c0 = 128 * half; c0 < 128 * half + 128; c0 += 32) {
        uint4 hv[4];  // H[p][c0 .. c0 + 31] (bf16)
#pragma unroll
        for (int q = 0; q < 4; ++q) hv[q] = hrow[c0 / 8 + q];
        uint32_t rp[32], ry[32];
        tmem_load_32cols(t_row + c0, rp);
        tmem_load_32cols(t_row + 256 + c0, ry);
        tmem_load_wait();
        const uint32_t hw[16] = {hv[0].x, hv[0].y, hv[0].z, hv[0].w, hv[1].x, hv[1].y,
                                 hv[1].z, hv[1].w, hv[2].x, hv[2].y, hv[2].z, hv[2].w,
                                 hv[3].x, hv[3].y, hv[3].z, hv[3].w};
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const float h = (e & 1) ? bf_hi(hw[e >> 1]) : bf_lo(hw[e >> 1]);
          const float pn = 2.f * h - __uint_as_float(rp[e]);
          rp[e] = __float_as_uint(pn);
          ry[e] = __float_as_uint(pn + __uint_as_float(ry[e]));
        }
        if (!last) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint32_t pw[4], yw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int ia = 8 * g + 2 * e;
              const __nv_bfloat162 pz =
                  __floats2bfloat162_rn(__uint_as_float(rp[ia]), __uint_as_float(rp[ia + 1]));
              const __nv_bfloat162 yz =
                  __floats2bfloat162_rn(__uint_as_float(ry[ia]), __uint_as_float(ry[ia + 1]));
              pw[e] = *reinterpret_cast<const uint32_t*>(&pz);
              yw[e] = *reinterpret_cast<const uint32_t*>(&yz);
            }
            const int c = c0 + 8 * g;
            st_shared_v4(tP + op_off(row, c), pw[0], pw[1], pw[2], pw[3]);
            // Y[p][c..c+7] is row k = p, columns c of the MN tile of the CTA
            // that owns columns c (this one or the peer)
            st_cluster_v4(mnY[c >> 7] + mn_off(p, c & 127), yw[0], yw[1], yw[2], yw[3]);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) ry[e] = __float_as_uint(-__uint_as_float(ry[e]));
          stage_gq32(ry, c0, to_peer, own, cross);
        }
      }
      if (!last) {
        fence_proxy_async_all();  // P, Y (here and in the peer) -> the next MMAs
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(map_peer(smem_u32(readyE), 0));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // -D staged in both CTAs
  pack_dtheta(b, lb, qs.P, rank, lsb, a.nb, dtheta, gq_own, gq_cross);
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

bool cnp_pair_fits(int b, int k) {
  return k >= 1 && k <= 16 && b >= 32 && b <= 256 && 256 % b == 0;
}

cudaError_t cnp_build_pair(const float* theta, int n, int b, int k, __nv_bfloat16* blocks,
                           cudaStream_t stream) {
  if (!cnp_pair_fits(b, k) || n <= 0 || (static_cast<long long>(n) * b) % 256 != 0)
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
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(cnp_build_pair_k_kernel,
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
  cudaError_t e = k == 3 ? cudaLaunchKernelEx(&cfg, cnp_build_pair_kernel, a)
                         : cudaLaunchKernelEx(&cfg, cnp_build_pair_k_kernel, a, k);
  prof_end("cnp_build", stream);
  return e != cudaSuccess ? e : cudaGetLastError();
}


cudaError_t cnp_adjoint_pair(const CnpAdjointPairArgs& x, cudaStream_t stream) {
  const int b = x.b;
  if (!cnp_pair_fits(b, x.k) || x.n_a + x.n_b <= 0 ||
      (static_cast<long long>(x.n_a) * b) % 256 != 0 || (static_cast<long long>(x.n_b) * b) % 256 != 0)
    return cudaErrorInvalidValue;
  static bool attr_set[64] = {false};
  static std::mutex mu;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_set[dev]) {
      cudaError_t e = cudaFuncSetAttribute(cnp_adjoint_pair_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, kAdjSmem);
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(cnp_adjoint_pair_k_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kAdjSmem);
      if (e != cudaSuccess) return e;
      attr_set[dev] = true;
    }
  }
  CnpAdjArgs a;
  a.theta_a = x.theta_a;
  a.theta_b = x.theta_b;
  a.part_a = x.part_a;
  a.part_b = x.part_b;
  a.splits_a = x.splits_a;
  a.splits_b = x.splits_b;
  a.nsb_a = static_cast<int>(static_cast<long long>(x.n_a) * b / 256);
  a.nsb_b = static_cast<int>(static_cast<long long>(x.n_b) * b / 256);
  a.b = b;
  a.nb = 256 / b;
  a.hg = x.hg;
  a.dtheta_a = x.dtheta_a;
  a.dtheta_b = x.dtheta_b;
  a.status = device_status_ptr();
  const int nsb = a.nsb_a + a.nsb_b;
  // H's rows as K-major 64 x 128 boxes; 64 x 64 boxes for G = H^T read MN-major
  CUtensorMap tmH, tmHmn;
  if (!make_map(&tmH, x.hg, static_cast<long long>(nsb) * 256, 256, 256, 2, BK, BM) ||
      !make_map(&tmHmn, x.hg, static_cast<long long>(nsb) * 256, 256, 256, 2, 64, BK))
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * nsb));
  cfg.blockDim = dim3(kCnpThreads);
  cfg.dynamicSmemBytes = kAdjSmem;
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
  // the token sums first, on all SMs
  const long long sum_items = static_cast<long long>(nsb) * 256 * 32;
  // two CTAs per SM: the adjoint's CTAs (which it lets launch at once) still
  // fit beside them by registers and start their theta-only phase
  const long long sum_cap = static_cast<long long>(sm_count()) * 2;
  const long long sum_blocks = (sum_items + 255) / 256;
  prof_begin("cnp_sums", stream);
  cudaError_t e = launch_pdl(cnp_sum_partials_kernel,
                             dim3(static_cast<unsigned>(sum_blocks < sum_cap ? sum_blocks : sum_cap)),
                             dim3(256), 0, stream, a);
  prof_end("cnp_sums", stream);
  if (e != cudaSuccess) return e;
  prof_begin("cnp_adjoint", stream);
  e = x.k == 3 ? cudaLaunchKernelEx(&cfg, cnp_adjoint_pair_kernel, tmH, tmHmn, a)
                            : cudaLaunchKernelEx(&cfg, cnp_adjoint_pair_k_kernel, tmH, tmHmn, a, x.k);
  prof_end("cnp_adjoint", stream);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace poetx
