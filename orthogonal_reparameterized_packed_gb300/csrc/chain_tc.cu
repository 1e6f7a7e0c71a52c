// The b x b product chains of the block build and of its adjoint, each run
// as ONE cooperative persistent launch.
//
// A chain is a short program of phases executed by every CTA in order:
//   elementwise phases  (unpack theta -> Q; split-K sums of the token-wise
//                        block gradients; I + Q; skew pack)  run by the four
//                        epilogue warps of every CTA, grid-stride;
//   product phases      1 or 2 problems  out = epi(A_g * B_g^T)  over all
//                        b x b blocks g, as 128 x 128 tcgen05 tiles
//                        (A K-major, B MN-major; both read by TMA from the
//                        row-major [n][b][b] stacks).
// Phase p+1 may read anything phase p wrote, so phases are separated by a
// grid barrier: every CTA bumps a global counter when its epilogue warps are
// done with phase p, and producers / epilogues of phase p+1 wait until the
// counter reaches (p+1) * gridDim.x.  The launch is cooperative, so all CTAs
// are resident; every wait is bounded (2 s) and records POETX_ERR_TIMEOUT.
//
// This is the "one fused kernel for Q^2, Q^3, Q^4" of the pages' CNP step,
// extended to the adjoint: a 256 x 256 bf16 operand pair does not fit one
// SM, so the chain runs on all SMs and synchronises between powers.
#include <algorithm>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace poetx {

namespace {

constexpr int CH_STAGES = 4;
constexpr int CH_THREADS = 192;
constexpr int CH_BN = 128;
constexpr int CH_A_BYTES = BM * BK * 2;     // 16 KB
constexpr int CH_B_BYTES = CH_BN * BK * 2;  // 16 KB
constexpr int CH_SMEM = 1024 + CH_STAGES * (CH_A_BYTES + CH_B_BYTES) + 256;
constexpr uint32_t CH_TMEM_COLS = 2 * CH_BN;

enum { OP_GEMM = 0, OP_UNPACK = 1, OP_PREP_BWD = 2, OP_IDENTITY = 3, OP_PACK = 4 };

constexpr int kChainMaxMaps = 40;
constexpr int kChainMaxPhases = 24;

struct ChainProd {
  int a_map, b_map;  // A: K-major box map, B: MN-major box map
  EpiArgs epi;
};

struct ChainPhase {
  int op;
  int nprod;
  ChainProd prod[2];
};

struct ChainParams {
  CUtensorMap maps[kChainMaxMaps];  // first member: keeps the maps 64-byte aligned
  ChainPhase phases[kChainMaxPhases];
  int nphases;
  int n, b, n_a;  // blocks, block size, blocks of the first side
  // elementwise operands
  const float* theta_a;
  const float* theta_b;
  float* q32;
  __nv_bfloat16* q16;
  const float* part_a;  // split-K partials [splits][nsb][S][S] of each side
  const float* part_b;
  int splits_a, splits_b, nsb_a, nsb_b, S;
  float* g32;  // reduced block gradients (fp32 + bf16)
  __nv_bfloat16* g16;
  const float* pack_A;
  const float* pack_B;
  float pack_sign;
  float* dtheta_a;
  float* dtheta_b;
  float* id32;
  __nv_bfloat16* id16;
  unsigned int* counter;
  int* status;
};

static_assert(sizeof(ChainParams) <= 32000, "chain parameters exceed the kernel parameter space");

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Wait until every CTA has finished the phases before `phase`.
__device__ bool grid_wait(const ChainParams& P, int phase, volatile int* abort) {
  const unsigned target = static_cast<unsigned>(phase) * gridDim.x;
  if (ld_acquire_u32(P.counter) >= target) return true;
  const unsigned long long t0 = global_timer_ns();
  while (true) {
    __nanosleep(64);
    if (ld_acquire_u32(P.counter) >= target) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      record_timeout(P.status, abort);
      return false;
    }
  }
}

__device__ __forceinline__ int packed_index(int i, int j, int b) {
  return i * b - (i * (i + 1)) / 2 + (j - i - 1);
}

// Elementwise phases, grid-stride over the n * b * b block entries.
__device__ void elementwise_phase(const ChainParams& P, int op, int tid, int nthreads) {
  const int b = P.b, bb = b * b, m = b * (b - 1) / 2;
  const int total = P.n * bb;
  for (int idx = tid; idx < total; idx += nthreads) {
    const int g = idx / bb;
    const int rem = idx - g * bb;
    const int i = rem / b;
    const int j = rem - i * b;
    const bool side_a = g < P.n_a;
    if (op == OP_UNPACK || op == OP_PREP_BWD) {
      const float* th = side_a ? P.theta_a + g * m : P.theta_b + (g - P.n_a) * m;
      float q = 0.f;
      if (i < j) q = th[packed_index(i, j, b)];
      else if (i > j) q = -th[packed_index(j, i, b)];
      P.q32[idx] = q;
      P.q16[idx] = __float2bfloat16_rn(q);
    }
    if (op == OP_PREP_BWD) {
      // diagonal b-block of superblock g / (S/b), summed over the K splits
      const int per = P.S / b;
      const int gl = side_a ? g : g - P.n_a;
      const int sb = gl / per;
      const int off = (gl - sb * per) * b;
      const float* part = side_a ? P.part_a : P.part_b;
      const int splits = side_a ? P.splits_a : P.splits_b;
      const long long stride = static_cast<long long>(side_a ? P.nsb_a : P.nsb_b) * P.S * P.S;
      const long long src = (static_cast<long long>(sb) * P.S + off + i) * P.S + off + j;
      float v = 0.f;
      for (int s = 0; s < splits; ++s) v += part[s * stride + src];
      P.g32[idx] = v;
      P.g16[idx] = __float2bfloat16_rn(v);
    }
    if (op == OP_IDENTITY) {
      const float v = P.q32[idx] + (i == j ? 1.f : 0.f);
      if (P.id32 != nullptr) P.id32[idx] = v;
      if (P.id16 != nullptr) P.id16[idx] = __float2bfloat16_rn(v);
    }
    if (op == OP_PACK && i < j) {
      const int ji = g * bb + j * b + i;
      float v = P.pack_A[idx] - P.pack_A[ji];
      if (P.pack_B != nullptr) v += P.pack_B[idx] - P.pack_B[ji];
      v *= P.pack_sign;
      if (side_a) P.dtheta_a[g * m + packed_index(i, j, b)] = v;
      else P.dtheta_b[(g - P.n_a) * m + packed_index(i, j, b)] = v;
    }
  }
}

__device__ __forceinline__ void decode_chain_tile(int t, int n, int mtl, int ntl, int& prod,
                                                  int& g, int& mt, int& nt) {
  const int per_prod = n * mtl * ntl;
  prod = t / per_prod;
  t -= prod * per_prod;
  g = t / (mtl * ntl);
  t -= g * mtl * ntl;
  mt = t / ntl;
  nt = t - mt * ntl;
}

__global__ void __launch_bounds__(CH_THREADS, 1) chain_kernel(const __grid_constant__ ChainParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + CH_STAGES * CH_A_BYTES;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(base + CH_STAGES * (CH_A_BYTES + CH_B_BYTES));
  uint64_t* empty_bar = full_bar + CH_STAGES;
  uint64_t* tfull_bar = empty_bar + CH_STAGES;  // [2]
  uint64_t* tempty_bar = tfull_bar + 2;         // [2]
  uint64_t* drain_bar = tempty_bar + 2;
  uint64_t* epi_done_bar = drain_bar + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(epi_done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int b = P.b;
  const int mtl = b / BM, ntl = b / CH_BN, ksteps = b / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < CH_STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], 4);
    }
    mbar_init(drain_bar, 1);
    mbar_init(epi_done_bar, 4);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, CH_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase_bit = 0;
      long long issued = 0;
      bool ok = true;
      for (int ph = 0; ph < P.nphases && ok; ++ph) {
        const ChainPhase& PH = P.phases[ph];
        if (PH.op != OP_GEMM) continue;
        if (!grid_wait(P, ph, abort_flag)) {
          ok = false;
          break;
        }
        fence_proxy_async_global();  // generic writes of earlier phases -> TMA reads
        const int tiles = PH.nprod * P.n * mtl * ntl;
        for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
          int prod, g, mt, nt;
          decode_chain_tile(t, P.n, mtl, ntl, prod, g, mt, nt);
          const CUtensorMap* ma = &P.maps[PH.prod[prod].a_map];
          const CUtensorMap* mb = &P.maps[PH.prod[prod].b_map];
          for (int ks = 0; ks < ksteps; ++ks) {
            if (!mbar_wait(&empty_bar[stage], phase_bit ^ 1, abort_flag)) {
              record_timeout(P.status, abort_flag);
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&full_bar[stage], CH_A_BYTES + CH_B_BYTES);
            uint8_t* a_dst = sA + stage * CH_A_BYTES;
            uint8_t* b_dst = sB + stage * CH_B_BYTES;
            tma_load_2d(a_dst, ma, &full_bar[stage], ks * BK, g * b + mt * BM);
            tma_load_2d(b_dst, mb, &full_bar[stage], nt * CH_BN, g * b + ks * BK);
            tma_load_2d(b_dst + 8192, mb, &full_bar[stage], nt * CH_BN + 64, g * b + ks * BK);
            ++issued;
            if (++stage == CH_STAGES) {
              stage = 0;
              phase_bit ^= 1;
            }
          }
        }
      }
      if (!ok) {
        const int outstanding = issued < CH_STAGES ? static_cast<int>(issued) : CH_STAGES;
        int st = stage;
        uint32_t pb = phase_bit;
        for (int i = 0; i < outstanding; ++i) {
          if (--st < 0) {
            st = CH_STAGES - 1;
            pb ^= 1;
          }
          const unsigned long long t0 = global_timer_ns();
          while (!mbar_try_wait(&full_bar[st], pb) && global_timer_ns() - t0 < 10000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------- MMA issuer
      constexpr uint32_t IDESC = instr_desc_bf16(BM, CH_BN, false, true);
      int stage = 0;
      uint32_t phase_bit = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, any_mma = false;
      for (int ph = 0; ph < P.nphases && ok; ++ph) {
        const ChainPhase& PH = P.phases[ph];
        if (PH.op != OP_GEMM) continue;
        const int tiles = PH.nprod * P.n * mtl * ntl;
        for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
          if (!mbar_wait(&tempty_bar[acc], acc_phase ^ 1, abort_flag)) {
            record_timeout(P.status, abort_flag);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * CH_BN);
          for (int ks = 0; ks < ksteps; ++ks) {
            if (!mbar_wait(&full_bar[stage], phase_bit, abort_flag)) {
              record_timeout(P.status, abort_flag);
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_base = smem_u32(sA + stage * CH_A_BYTES);
            const uint32_t b_base = smem_u32(sB + stage * CH_B_BYTES);
#pragma unroll
            for (int j = 0; j < BK / 16; ++j) {
              const uint64_t adesc = smem_desc_sw128(a_base + j * 32, 16, 1024);
              const uint64_t bdesc = smem_desc_sw128(b_base + j * 2048, 8192, 1024);
              umma_bf16(d_tmem, adesc, bdesc, IDESC, (ks > 0 || j > 0) ? 1u : 0u);
            }
            any_mma = true;
            umma_commit(&empty_bar[stage]);
            if (++stage == CH_STAGES) {
              stage = 0;
              phase_bit ^= 1;
            }
          }
          if (!ok) break;
          umma_commit(&tfull_bar[acc]);
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1;
        }
      }
      if (!ok && any_mma) {
        umma_commit(drain_bar);
        const unsigned long long t0 = global_timer_ns();
        while (!mbar_try_wait(drain_bar, 0) && global_timer_ns() - t0 < 10000000ull) {
        }
      }
    }
  } else {
    // ---------------------------------------------- epilogue / elementwise
    const int quarter = warp & 3;
    const int etid = blockIdx.x * 128 + (threadIdx.x - 64);
    const int ethreads = gridDim.x * 128;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int ph = 0; ph < P.nphases; ++ph) {
      const ChainPhase& PH = P.phases[ph];
      int ok = 1;
      if (ph > 0 && lane == 0) ok = grid_wait(P, ph, abort_flag) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (PH.op == OP_GEMM) {
        const int tiles = PH.nprod * P.n * mtl * ntl;
        for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
          int prod, g, mt, nt;
          decode_chain_tile(t, P.n, mtl, ntl, prod, g, mt, nt);
          const bool got = mbar_wait(&tfull_bar[acc], acc_phase, abort_flag);
          if (!__all_sync(0xffffffffu, got)) {  // the whole warp unwinds together
            record_timeout(P.status, abort_flag);
            ok = 0;
            break;
          }
          tc_fence_after();
          const uint32_t t_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                  static_cast<uint32_t>(acc * CH_BN);
          const int row = mt * BM + quarter * 32 + lane;
#pragma unroll 1
          for (int c0 = 0; c0 < CH_BN; c0 += 32) {
            uint32_t r[32];
            tmem_load_32cols(t_base + c0, r);
            tmem_load_wait();
            epilogue_row32(PH.prod[prod].epi, g, 0, row, nt * CH_BN + c0, r);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty_bar[acc]);
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1;
        }
        if (!ok) break;
      } else {
        elementwise_phase(P, PH.op, etid, ethreads);
      }
      // this warp is done with the phase; the first epilogue warp publishes
      // the CTA's completion once all four are
      __syncwarp();
      if (lane == 0) mbar_arrive(epi_done_bar);
      if (warp == 2 && lane == 0) {
        if (!mbar_wait(epi_done_bar, ph & 1, abort_flag)) {
          record_timeout(P.status, abort_flag);
          ok = 0;
        } else {
          __threadfence();
          atomicAdd(P.counter, 1u);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, CH_TMEM_COLS);
  }
}

// ------------------------------------------------------------- host side

// Map index of buffer `buf` used as a K-major A operand (box 64 x 128) or an
// MN-major B operand (box 64 x 64).
struct MapTable {
  ChainParams* P;
  int count = 0;
  bool ok = true;
  const void* ptrs[kChainMaxMaps / 2];
  int add(const void* buf, int n, int b) {  // returns the K-box index; MN-box = +1
    for (int i = 0; i < count; i += 2)
      if (ptrs[i / 2] == buf) return i;
    if (count + 2 > kChainMaxMaps) {
      ok = false;
      return 0;
    }
    const long long rows = static_cast<long long>(n) * b;
    ok = ok && make_map(&P->maps[count], buf, rows, b, b, 2, BK, BM);
    ok = ok && make_map(&P->maps[count + 1], buf, rows, b, b, 2, BK, 64);
    ptrs[count / 2] = buf;
    count += 2;
    return count - 2;
  }
};

EpiArgs chain_epi(int b) {
  EpiArgs e;
  e.ld = b;
  e.row_g = b;
  return e;
}

cudaError_t launch_chain(ChainParams& P, cudaStream_t stream) {
  static bool attr_set[64] = {false};
  static int max_ctas[64] = {0};
  static std::mutex mu;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_set[dev]) {
      cudaError_t e = cudaFuncSetAttribute(chain_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, CH_SMEM);
      if (e != cudaSuccess) return e;
      int per_sm = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, chain_kernel, CH_THREADS,
                                                        CH_SMEM);
      if (e != cudaSuccess) return e;
      max_ctas[dev] = per_sm * sm_count();
      attr_set[dev] = true;
    }
  }
  int most_tiles = 1;
  for (int ph = 0; ph < P.nphases; ++ph)
    if (P.phases[ph].op == OP_GEMM)
      most_tiles = std::max(most_tiles, P.phases[ph].nprod * P.n * (P.b / BM) * (P.b / CH_BN));
  const int grid = std::min(most_tiles, std::min(max_ctas[dev], sm_count()));
  if (grid < 1) return cudaErrorLaunchOutOfResources;
  P.status = device_status_ptr();
  cudaError_t e = cudaMemsetAsync(P.counter, 0, sizeof(unsigned int), stream);
  if (e != cudaSuccess) return e;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(CH_THREADS);
  cfg.dynamicSmemBytes = CH_SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs resident: they wait on one another
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_begin("chain", stream);
  e = cudaLaunchKernelEx(&cfg, chain_kernel, P);
  prof_end("chain", stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t chain_build(const float* theta, int n, int b, int k, float* q32, __nv_bfloat16* q16,
                        __nv_bfloat16* e16a, __nv_bfloat16* e16b, unsigned int* counter,
                        __nv_bfloat16* blocks, cudaStream_t stream) {
  if (k > kChainMaxK || b % CH_BN != 0) return cudaErrorInvalidValue;
  static ChainParams P;  // large: kept off the stack; calls are host-serialised below
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  P = ChainParams();
  P.n = n;
  P.b = b;
  P.n_a = n;
  P.theta_a = theta;
  P.q32 = q32;
  P.q16 = q16;
  P.id16 = blocks;
  P.counter = counter;
  MapTable maps{&P};
  int ph = 0;
  P.phases[ph++].op = OP_UNPACK;
  if (k == 0) {
    P.phases[ph++].op = OP_IDENTITY;
  } else {
    const int q_map = maps.add(q16, n, b);
    int cur_map = q_map;  // E_{k+1} = Q
    __nv_bfloat16* ebuf[2] = {e16a, e16b};
    int nxt = 0;
    for (int i = k; i >= 1; --i) {
      ChainPhase& PH = P.phases[ph++];
      PH.op = OP_GEMM;
      PH.nprod = 1;
      PH.prod[0].a_map = q_map;        // Q, K-major
      PH.prod[0].b_map = cur_map + 1;  // E_{i+1}, MN-major: B[n][kk] = E[kk][n]
      EpiArgs e = chain_epi(b);
      e.X = q32;  // + 2 Q
      e.beta = 2.f;
      if (i == 1) {
        e.delta = 1.f;  // + I
        e.out_bf16 = blocks;
      } else {
        e.out_bf16 = ebuf[nxt];
        cur_map = maps.add(ebuf[nxt], n, b);
        nxt ^= 1;
      }
      PH.prod[0].epi = e;
    }
  }
  P.nphases = ph;
  if (!maps.ok) return cudaErrorInvalidValue;
  return launch_chain(P, stream);
}

cudaError_t chain_adjoint(const ChainAdjointArgs& a, cudaStream_t stream) {
  const int k = a.k, b = a.b, n = a.n_a + a.n_b;
  if (k > kChainMaxK || b % CH_BN != 0) return cudaErrorInvalidValue;
  static ChainParams P;
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  P = ChainParams();
  P.n = n;
  P.b = b;
  P.n_a = a.n_a;
  P.theta_a = a.theta_a;
  P.theta_b = a.theta_b;
  P.q32 = a.q32;
  P.q16 = a.q16;
  P.part_a = a.part_a;
  P.part_b = a.part_b;
  P.splits_a = a.splits_a;
  P.splits_b = a.splits_b;
  P.nsb_a = a.nsb_a;
  P.nsb_b = a.nsb_b;
  P.S = a.S;
  P.g32 = a.f32[0];
  P.g16 = a.f16[0];
  P.dtheta_a = a.dtheta_a;
  P.dtheta_b = a.dtheta_b;
  P.pack_sign = -1.f;  // D = dQ^T: pack(dQ - dQ^T) = -pack(D - D^T)
  P.counter = a.counter;
  MapTable maps{&P};
  int ph = 0;
  P.phases[ph++].op = OP_PREP_BWD;  // Q, and F_1 = G^T from the split-K partials
  const int q_map = maps.add(a.q16, n, b);
  int e_map[kChainMaxK + 2];
  e_map[k + 1] = q_map;
  // E_i = 2Q + Q E_{i+1}, i = k .. 2
  for (int i = k; i >= 2; --i) {
    ChainPhase& PH = P.phases[ph++];
    PH.op = OP_GEMM;
    PH.nprod = 1;
    PH.prod[0].a_map = q_map;
    PH.prod[0].b_map = e_map[i + 1] + 1;
    EpiArgs e = chain_epi(b);
    e.X = a.q32;
    e.beta = 2.f;
    e.out_bf16 = a.e16[i];
    PH.prod[0].epi = e;
    e_map[i] = maps.add(a.e16[i], n, b);
  }
  // transposed reverse sweep: D += 2 F_i + E_{i+1} F_i,  F_{i+1} = F_i Q
  int cur = 0;
  for (int i = 1; i <= k; ++i) {
    ChainPhase& PH = P.phases[ph++];
    PH.op = OP_GEMM;
    PH.nprod = 2;
    const int f_map = maps.add(a.f16[cur], n, b);
    PH.prod[0].a_map = e_map[i + 1];  // E_{i+1}, K-major
    PH.prod[0].b_map = f_map + 1;     // B[n][kk] = F_i[kk][n]
    EpiArgs e0 = chain_epi(b);
    if (i > 1) {
      e0.X = a.d32;
      e0.beta = 1.f;
    }
    e0.Y = a.f32[cur];
    e0.gamma = 2.f;
    e0.out_f32 = a.d32;
    PH.prod[0].epi = e0;
    PH.prod[1].a_map = f_map;      // F_i, K-major
    PH.prod[1].b_map = q_map + 1;  // B[n][kk] = Q[kk][n]
    EpiArgs e1 = chain_epi(b);
    e1.out_f32 = a.f32[1 - cur];
    e1.out_bf16 = a.f16[1 - cur];
    PH.prod[1].epi = e1;
    cur = 1 - cur;
  }
  ChainPhase& PK = P.phases[ph++];
  PK.op = OP_PACK;
  if (k == 0) {
    P.pack_A = a.f32[0];
    P.pack_B = nullptr;
  } else {
    P.pack_A = a.d32;
    P.pack_B = a.f32[cur];  // F_{k+1}
  }
  P.nphases = ph;
  if (!maps.ok) return cudaErrorInvalidValue;
  return launch_chain(P, stream);
}

}  // namespace poetx
