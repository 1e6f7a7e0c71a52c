// Tensor-core contraction engine for sm_103a: C = A * B^T per batch, bf16
// operands staged by TMA into 128-byte-swizzled shared memory, tcgen05.mma
// accumulating in TMEM, fp32 epilogue straight from TMEM.
//
// One persistent CTA per SM, warp-specialised:
//   warp 0      TMA producer (one elected lane), STAGES-deep smem ring
//   warp 1      TMEM allocator + MMA issuer (one elected lane)
//   warps 2..5  epilogue: TMEM -> registers -> EpiArgs -> global
// Two TMEM accumulators (2 x BN fp32 columns) let the epilogue of tile i
// overlap the main loop of tile i+1.  Every barrier wait is bounded: on
// expiry the CTA records POETX_ERR_TIMEOUT, drains what it issued, frees
// TMEM and returns.
//
// Every contraction of the layer maps onto this engine: the W0 GEMM and its
// transpose, the block-diagonal transforms (batch = diagonal block, K window
// = that block's features), the per-block outer products summed over tokens
// (split-K over tokens), and the b x b products of the block builder and its
// adjoint.
#include <algorithm>
#include <cstdio>

#include "internal.h"
#include "ptx.cuh"

namespace poetx {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;  // one 128-byte swizzle row of bf16
constexpr int STAGES = 4;
constexpr int NUM_THREADS = 192;
constexpr int kStatusTimeout = 5;  // POETX_ERR_TIMEOUT

template <int BN>
struct TcShape {
  static constexpr int A_BYTES = BM * BK * 2;  // 16 KB
  static constexpr int B_BYTES = BN * BK * 2;  // 16 or 32 KB
  static constexpr int SMEM = 1024 + STAGES * (A_BYTES + B_BYTES) + 256;
  static constexpr uint32_t TMEM_COLS = 2 * BN;
};

struct TcKernelArgs {
  int m_tiles, n_tiles, splits, batches;
  int k_steps_total, k_steps_per_split;
  int a_mn_per_g, a_k_per_g, b_mn_per_g, b_k_per_g;
  EpiArgs epi;
  int* status;
};

__device__ __forceinline__ void record_timeout(int* status, volatile int* abort) {
  atomicCAS(status, 0, kStatusTimeout);
  *abort = 1;
}

// Apply the epilogue to 32 consecutive accumulator columns of one row.
__device__ __forceinline__ void epilogue_row32(const EpiArgs& e, int g, int s, int row, int col0,
                                               const uint32_t (&r)[32]) {
  if (row >= e.row_limit) return;
  const long long off = (long long)g * e.g_off + (long long)s * e.s_off +
                        (long long)row * e.ld + col0;
  float v[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = e.alpha * __uint_as_float(r[j]);
  if (e.X != nullptr) {
    const float4* xp = reinterpret_cast<const float4*>(e.X + off);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 t = xp[q];
      v[4 * q + 0] += e.beta * t.x;
      v[4 * q + 1] += e.beta * t.y;
      v[4 * q + 2] += e.beta * t.z;
      v[4 * q + 3] += e.beta * t.w;
    }
  }
  if (e.Y != nullptr) {
    const float4* yp = reinterpret_cast<const float4*>(e.Y + off);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 t = yp[q];
      v[4 * q + 0] += e.gamma * t.x;
      v[4 * q + 1] += e.gamma * t.y;
      v[4 * q + 2] += e.gamma * t.z;
      v[4 * q + 3] += e.gamma * t.w;
    }
  }
  if (e.delta != 0.f) {
    const int dj = row - col0;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j == dj) v[j] += e.delta;
  }
  if (e.out_f32 != nullptr) {
    float4* op = reinterpret_cast<float4*>(e.out_f32 + off);
#pragma unroll
    for (int q = 0; q < 8; ++q)
      op[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  }
  if (e.out_bf16 != nullptr) {
    uint4* op = reinterpret_cast<uint4*>(e.out_bf16 + off);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t w[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        __nv_bfloat162 p2 = __floats2bfloat162_rn(v[8 * q + 2 * h], v[8 * q + 2 * h + 1]);
        w[h] = *reinterpret_cast<uint32_t*>(&p2);
      }
      op[q] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

template <bool A_MN, bool B_MN, int BN>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB, const TcKernelArgs p) {
  using S = TcShape<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + STAGES * S::A_BYTES;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(sB + STAGES * S::B_BYTES);
  uint64_t* empty_bar = full_bar + STAGES;
  uint64_t* tfull_bar = empty_bar + STAGES;  // [2]
  uint64_t* tempty_bar = tfull_bar + 2;      // [2]
  uint64_t* drain_bar = tempty_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const int num_tiles = p.batches * p.splits * p.m_tiles * p.n_tiles;

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
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, S::TMEM_COLS);
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
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        int t = tile;
        const int nt = t % p.n_tiles;
        t /= p.n_tiles;
        const int mt = t % p.m_tiles;
        t /= p.m_tiles;
        const int sp = t % p.splits;
        const int g = t / p.splits;
        const int ks0 = sp * p.k_steps_per_split;
        const int ks1 = min(ks0 + p.k_steps_per_split, p.k_steps_total);
        const int a_mn = g * p.a_mn_per_g + mt * BM;
        const int b_mn = g * p.b_mn_per_g + nt * BN;
        for (int ks = ks0; ks < ks1; ++ks) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1, abort_flag)) {
            record_timeout(p.status, abort_flag);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full_bar[stage], S::A_BYTES + S::B_BYTES);
          const int a_k = g * p.a_k_per_g + ks * BK;
          const int b_k = g * p.b_k_per_g + ks * BK;
          uint8_t* a_dst = sA + stage * S::A_BYTES;
          uint8_t* b_dst = sB + stage * S::B_BYTES;
          if (!A_MN) {
            tma_load_2d(a_dst, &tmA, &full_bar[stage], a_k, a_mn);
          } else {
            tma_load_2d(a_dst, &tmA, &full_bar[stage], a_mn, a_k);
            tma_load_2d(a_dst + 8192, &tmA, &full_bar[stage], a_mn + 64, a_k);
          }
          if (!B_MN) {
            tma_load_2d(b_dst, &tmB, &full_bar[stage], b_k, b_mn);
          } else {
#pragma unroll
            for (int c = 0; c < BN / 64; ++c)
              tma_load_2d(b_dst + c * 8192, &tmB, &full_bar[stage], b_mn + 64 * c, b_k);
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
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
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        int t = tile / (p.n_tiles * p.m_tiles);
        const int sp = t % p.splits;
        const int ks0 = sp * p.k_steps_per_split;
        const int ks1 = min(ks0 + p.k_steps_per_split, p.k_steps_total);
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
          const uint32_t b_base = smem_u32(sB + stage * S::B_BYTES);
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
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
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
    const int row_in_tile = quarter * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      int t = tile;
      const int nt = t % p.n_tiles;
      t /= p.n_tiles;
      const int mt = t % p.m_tiles;
      t /= p.m_tiles;
      const int sp = t % p.splits;
      const int g = t / p.splits;
      if (!mbar_wait(&tfull_bar[acc], acc_phase, abort_flag)) {
        record_timeout(p.status, abort_flag);
        break;
      }
      tc_fence_after();
      const int row = mt * BM + row_in_tile;
      const uint32_t t_base =
          tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * BN);
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t r[32];
        tmem_load_32cols(t_base + c0, r);
        tmem_load_wait();
        epilogue_row32(p.epi, g, sp, row, nt * BN + c0, r);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty_bar[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, S::TMEM_COLS);
  }
}

// ------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// 2-D bf16 map over a row-major array, box = box_cols x box_rows, 128B swizzle.
bool make_map(CUtensorMap* map, const TcOperand& op, int box_cols, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(op.cols), static_cast<cuuint64_t>(op.rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(op.pitch) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(op.ptr), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <bool A_MN, bool B_MN, int BN>
cudaError_t launch_tc(const TcGemm& g, cudaStream_t stream) {
  using S = TcShape<BN>;
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<A_MN, B_MN, BN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  CUtensorMap tmA, tmB;
  if (!make_map(&tmA, g.A, 64, A_MN ? 64 : BM)) return cudaErrorInvalidValue;
  if (!make_map(&tmB, g.B, 64, B_MN ? 64 : BN)) return cudaErrorInvalidValue;

  TcKernelArgs p;
  p.m_tiles = (g.M + BM - 1) / BM;
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
  p.status = device_status_ptr();
  const long long tiles = static_cast<long long>(p.batches) * p.splits * p.m_tiles * p.n_tiles;
  if (tiles <= 0) return cudaSuccess;
  const int grid = static_cast<int>(std::min<long long>(tiles, sm_count()));
  prof_begin(g.tag, stream);
  tc_gemm_kernel<A_MN, B_MN, BN><<<grid, NUM_THREADS, S::SMEM, stream>>>(tmA, tmB, p);
  prof_end(g.tag, stream);
  return cudaGetLastError();
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
  if (g.BN == 256) {
    if (!a && !b) return launch_tc<false, false, 256>(g, stream);
    if (!a && b) return launch_tc<false, true, 256>(g, stream);
    if (a && b) return launch_tc<true, true, 256>(g, stream);
  } else {
    if (!a && !b) return launch_tc<false, false, 128>(g, stream);
    if (!a && b) return launch_tc<false, true, 128>(g, stream);
    if (a && b) return launch_tc<true, true, 128>(g, stream);
  }
  return cudaErrorInvalidValue;  // (MN, K) is not used by the layer
}

}  // namespace poetx
