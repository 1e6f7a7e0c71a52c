// The b x b product chains of the block build and of its adjoint, each run
// as ONE cooperative persistent launch of product phases.
//
// Phase p computes 1 or 2 products over all b x b blocks g, each a sum of up
// to three MMA terms  sum_t A_t(g) * B_t(g)^T  (A K-major, B MN-major, read
// by TMA from the row-major [n][b][b] stacks or from a constant b x b
// matrix), as 128 x 128 tcgen05 tiles.  Addends are MMA terms too
// (2Q = Q_hi * 2I + Q_lo * 2I, 2F = F * 2I), so epilogues only store.  The
// adjoint's running sum D stays in TMEM across its phases: each CTA owns the
// same D tiles in every phase.  The elementwise steps around a chain (theta
// -> Q, split-K sums, skew pack) are separate, massively parallel tiled
// kernels (kernels_simt.cu).
//
// Phase p+1 reads what phase p wrote, so a grid barrier separates phases:
// each CTA bumps counter[p] when its epilogue warps have stored phase p, and
// producers of phase p+1 wait until counter[p] == gridDim.x.  One counter per
// phase: a CTA without tiles finishes later phases at once, and its early
// arrivals must not count towards an earlier phase.
// The launch is cooperative (all CTAs resident); every wait is bounded (2 s)
// and records POETX_ERR_TIMEOUT.  The counters are zeroed by the tiled prep
// kernel that always runs right before a chain.
//
// This is the pages' "Q^2, Q^3, Q^4 in one fused kernel" of the CNP step,
// extended to the adjoint; a 256 x 256 bf16 operand pair does not fit one
// SM, so the chain spans all SMs and synchronises between powers.
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
constexpr int CH_BARRIER_BYTES = 512;
constexpr int CH_SMEM = 1024 + CH_STAGES * (CH_A_BYTES + CH_B_BYTES) + CH_BARRIER_BYTES;
constexpr uint32_t CH_TMEM_COLS = 512;  // 2 rotating accumulators + 2 persistent D slots
constexpr int kMaxDSlots = 2;

enum { PROD_STORE = 0, PROD_ACC = 1, PROD_ACC_STORE = 2 };

constexpr int kChainMaxMaps = 48;
constexpr int kChainMaxTerms = 5;

struct ChainTerm {
  int a_map, b_map;  // A: K-major box map, B: MN-major box map
  int b_batched;     // B rows offset by g * b (0: one constant b x b matrix)
  int diag;          // B is diagonal (2I): only the K steps of the tile's own columns count
  int dep;           // lazy phases: the phase whose outputs this term reads (-1: none)
};

// K steps [k0, k1) of a term for output column tile nt
__device__ __forceinline__ void term_ksteps(const ChainTerm& T, int nt, int ksteps, int& k0,
                                            int& k1) {
  k0 = T.diag ? nt * (CH_BN / BK) : 0;
  k1 = T.diag ? k0 + CH_BN / BK : ksteps;
}

struct ChainProd {
  int nterms;
  ChainTerm term[kChainMaxTerms];
  int mode;       // PROD_STORE / PROD_ACC / PROD_ACC_STORE
  int first_acc;  // ACC modes: this phase initialises the persistent slot
  EpiArgs epi;    // stores only: alpha, delta, out_f32 / out_bf16
};

struct ChainPhase {
  int nprod;
  // lazy: the producer waits for each term's own dependency instead of for
  // the previous phase, so terms that read only the inputs (listed first)
  // load and multiply while the grid barrier is still open.  Only for phases
  // that overwrite nothing a running phase still reads.
  int lazy;
  ChainProd prod[2];
};

struct ChainParams {
  CUtensorMap maps[kChainMaxMaps];  // first member: keeps the maps 64-byte aligned
  ChainPhase phases[kChainMaxPhases];
  int nphases;
  int n, b;  // blocks, block size
  unsigned int* counter;  // [kChainMaxPhases] per-phase arrival counts
  int* status;
};

static_assert(sizeof(ChainParams) <= 32000, "chain parameters exceed the kernel parameter space");
static_assert((2 * CH_STAGES + 4 + kMaxDSlots + 1 + kChainMaxPhases) * 8 + 8 <= CH_BARRIER_BYTES,
              "chain barriers exceed their shared-memory area");

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}


// Wait until every CTA has finished phase `phase - 1`.
__device__ bool grid_wait(const ChainParams& P, int phase, volatile int* abort) {
  if (phase == 0) return true;
  const unsigned* c = P.counter + (phase - 1);
  const unsigned target = gridDim.x;
  if (ld_acquire_u32(c) >= target) return true;
  const unsigned long long t0 = global_timer_ns();
  while (true) {
    __nanosleep(100);
    if (ld_acquire_u32(c) >= target) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      record_timeout(P.status, abort);
      return false;
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
  uint64_t* dfull_bar = tempty_bar + 2;         // [kMaxDSlots]
  uint64_t* drain_bar = dfull_bar + kMaxDSlots;
  // one per phase, each completed once: epilogue warps of an idle CTA run
  // ahead through the phases, so a reused barrier would mix their arrivals
  uint64_t* epi_done_bar = drain_bar + 1;  // [kChainMaxPhases]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(epi_done_bar + kChainMaxPhases);
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
    for (int d = 0; d < kMaxDSlots; ++d) mbar_init(&dfull_bar[d], 1);
    mbar_init(drain_bar, 1);
    for (int q = 0; q < kChainMaxPhases; ++q) mbar_init(&epi_done_bar[q], 4);
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
  pdl_wait();
  pdl_trigger();  // the kernel after the chain may start its prologue

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase_bit = 0;
      long long issued = 0;
      bool ok = true;
      int waited = 0;  // phases known complete on the whole grid
      for (int ph = 0; ph < P.nphases && ok; ++ph) {
        const ChainPhase& PH = P.phases[ph];
        if (!PH.lazy && ph > waited) {
          if (!grid_wait(P, ph, abort_flag)) {
            ok = false;
            break;
          }
          waited = ph;
          fence_proxy_async_global();  // generic writes of earlier phases -> TMA reads
        }
        const int tiles = PH.nprod * P.n * mtl * ntl;
        for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
          int prod, g, mt, nt;
          decode_chain_tile(t, P.n, mtl, ntl, prod, g, mt, nt);
          const ChainProd& PR = PH.prod[prod];
          for (int term = 0; term < PR.nterms && ok; ++term) {
            if (PH.lazy && PR.term[term].dep + 1 > waited) {
              if (!grid_wait(P, PR.term[term].dep + 1, abort_flag)) {
                ok = false;
                break;
              }
              waited = PR.term[term].dep + 1;
              fence_proxy_async_global();
            }
            const CUtensorMap* ma = &P.maps[PR.term[term].a_map];
            const CUtensorMap* mb = &P.maps[PR.term[term].b_map];
            const int b_row0 = PR.term[term].b_batched ? g * b : 0;
            int k0, k1;
            term_ksteps(PR.term[term], nt, ksteps, k0, k1);
            for (int ks = k0; ks < k1; ++ks) {
              if (!mbar_wait(&empty_bar[stage], phase_bit ^ 1, abort_flag)) {
                record_timeout(P.status, abort_flag);
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(&full_bar[stage], CH_A_BYTES + CH_B_BYTES);
              uint8_t* a_dst = sA + stage * CH_A_BYTES;
              uint8_t* b_dst = sB + stage * CH_B_BYTES;
              tma_load_2d(a_dst, ma, &full_bar[stage], ks * BK, g * b + mt * BM);
              tma_load_2d(b_dst, mb, &full_bar[stage], nt * CH_BN, b_row0 + ks * BK);
              tma_load_2d(b_dst + 8192, mb, &full_bar[stage], nt * CH_BN + 64, b_row0 + ks * BK);
              ++issued;
              if (++stage == CH_STAGES) {
                stage = 0;
                phase_bit ^= 1;
              }
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
        const int tiles = PH.nprod * P.n * mtl * ntl;
        for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
          int prod, g, mt, nt;
          decode_chain_tile(t, P.n, mtl, ntl, prod, g, mt, nt);
          const ChainProd& PR = PH.prod[prod];
          const bool persistent = PR.mode != PROD_STORE;
          const int dslot = t / gridDim.x;  // same tile -> same CTA and slot in every phase
          uint32_t d_tmem;
          if (persistent) {
            d_tmem = tmem_base + 256u + static_cast<uint32_t>(dslot * CH_BN);
          } else {
            if (!mbar_wait(&tempty_bar[acc], acc_phase ^ 1, abort_flag)) {
              record_timeout(P.status, abort_flag);
              ok = false;
              break;
            }
            tc_fence_after();
            d_tmem = tmem_base + static_cast<uint32_t>(acc * CH_BN);
          }
          bool fresh = !persistent || PR.first_acc;
          for (int term = 0; term < PR.nterms && ok; ++term) {
            int k0, k1;
            term_ksteps(PR.term[term], nt, ksteps, k0, k1);
            for (int ks = k0; ks < k1; ++ks) {
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
                umma_bf16(d_tmem, adesc, bdesc, IDESC, fresh ? 0u : 1u);
                fresh = false;
              }
              any_mma = true;
              umma_commit(&empty_bar[stage]);
              if (++stage == CH_STAGES) {
                stage = 0;
                phase_bit ^= 1;
              }
            }
          }
          if (!ok) break;
          if (!persistent) {
            umma_commit(&tfull_bar[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1;
          } else if (PR.mode == PROD_ACC_STORE) {
            umma_commit(&dfull_bar[dslot]);  // the running sum is final
          }
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
    // ----------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int ph = 0; ph < P.nphases; ++ph) {
      const ChainPhase& PH = P.phases[ph];
      bool ok = true;
      const int tiles = PH.nprod * P.n * mtl * ntl;
      for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
        int prod, g, mt, nt;
        decode_chain_tile(t, P.n, mtl, ntl, prod, g, mt, nt);
        const ChainProd& PR = PH.prod[prod];
        if (PR.mode == PROD_ACC) continue;  // the running sum stays in TMEM
        const int dslot = t / gridDim.x;
        const bool got = PR.mode == PROD_STORE ? mbar_wait(&tfull_bar[acc], acc_phase, abort_flag)
                                               : mbar_wait(&dfull_bar[dslot], 0, abort_flag);
        if (!__all_sync(0xffffffffu, got)) {
          record_timeout(P.status, abort_flag);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t col = PR.mode == PROD_STORE ? static_cast<uint32_t>(acc * CH_BN)
                                                   : 256u + static_cast<uint32_t>(dslot * CH_BN);
        const uint32_t t_base = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + col;
        const int row = mt * BM + quarter * 32 + lane;
#pragma unroll 1
        for (int c0 = 0; c0 < CH_BN; c0 += 32) {
          uint32_t r[32];
          tmem_load_32cols(t_base + c0, r);
          tmem_load_wait();
          epilogue_row32(PR.epi, g, 0, row, nt * CH_BN + c0, r);
        }
        if (PR.mode == PROD_STORE) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty_bar[acc]);
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1;
        }
      }
      if (!ok) break;
      if (ph + 1 == P.nphases) break;  // nobody waits on the last phase
      // this warp has stored the phase; warp 2 publishes the CTA's completion
      // once all four epilogue warps have.  The next phase reads these
      // stores through TMA (the async proxy): each writing thread orders its
      // generic-proxy stores before that with a proxy fence.
      fence_proxy_async_global();
      __syncwarp();
      if (lane == 0) mbar_arrive(&epi_done_bar[ph]);
      if (warp == 2) {
        bool done = true;
        if (lane == 0) {
          done = mbar_wait(&epi_done_bar[ph], 0, abort_flag);
          if (done) {
            __threadfence();
            atomicAdd(P.counter + ph, 1u);
          } else {
            record_timeout(P.status, abort_flag);
          }
        }
        if (__shfl_sync(0xffffffffu, done ? 1 : 0, 0) == 0) break;
      }
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

// Two maps per buffer: K-major box (64 x 128) for A, MN-major box (64 x 64)
// for B; `rows` rows of b columns.
struct MapTable {
  ChainParams* P;
  int count = 0;
  bool ok = true;
  const void* ptrs[kChainMaxMaps / 2] = {};
  int add(const void* buf, long long rows, int b) {  // returns the K-box index; MN-box = +1
    for (int i = 0; i < count; i += 2)
      if (ptrs[i / 2] == buf) return i;
    if (count + 2 > kChainMaxMaps) {
      ok = false;
      return 0;
    }
    ok = ok && make_map(&P->maps[count], buf, rows, b, b, 2, BK, BM);
    ok = ok && make_map(&P->maps[count + 1], buf, rows, b, b, 2, BK, 64);
    ptrs[count / 2] = buf;
    count += 2;
    return count - 2;
  }
};

ChainTerm term(int a_map, int b_map, bool b_batched) {
  ChainTerm t;
  t.a_map = a_map;
  t.b_map = b_map + 1;  // MN-major box
  t.b_batched = b_batched ? 1 : 0;
  t.diag = 0;
  t.dep = -1;
  return t;
}

ChainTerm dep_on(ChainTerm t, int phase) {
  t.dep = phase;
  return t;
}

// A times the constant 2I: of the K sum only the tile's own column range is non-zero
ChainTerm term_2i(int a_map, int two_map) {
  ChainTerm t = term(a_map, two_map, false);
  t.diag = 1;
  return t;
}

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
  const int grid = std::min(max_ctas[dev], sm_count());
  if (grid < 1) return cudaErrorLaunchOutOfResources;
  // every persistent D tile needs a slot in its CTA
  for (int ph = 0; ph < P.nphases; ++ph)
    for (int q = 0; q < P.phases[ph].nprod; ++q)
      if (P.phases[ph].prod[q].mode != PROD_STORE) {
        const int tiles = P.n * (P.b / BM) * (P.b / CH_BN);
        if (q != 0 || (tiles + grid - 1) / grid > kMaxDSlots) return cudaErrorInvalidValue;
      }
  P.status = device_status_ptr();
  cudaError_t e;

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

std::mutex g_chain_mu;
ChainParams g_chain_params;  // large: kept off the stack; launches are host-serialised

}  // namespace

bool chain_fits(int n, int b, int k) {
  if (k < 1 || k > kChainMaxK || b % CH_BN != 0) return false;
  const int tiles = n * (b / BM) * (b / CH_BN);
  return (tiles + sm_count() - 1) / sm_count() <= kMaxDSlots;
}

cudaError_t chain_build(const ChainBuildArgs& a, cudaStream_t stream) {
  const int n = a.n, b = a.b, k = a.k;
  if (!chain_fits(n, b, k)) return cudaErrorInvalidValue;
  PrepTilesArgs pa;  // Q as bf16 hi + lo parts, and 2I
  pa.n_a = n;
  pa.b = b;
  pa.theta_a = a.theta;
  pa.q_hi = a.q_hi;
  pa.q_lo = a.q_lo;
  pa.q_x2 = k == 3 ? a.e16[1] : nullptr;  // 2 Q_hi for the two-phase k = 3 build
  pa.two_i = a.two_i;
  pa.zero_words = a.counter;
  pa.n_zero_words = kChainMaxPhases;
  cudaError_t e = launch_prep_tiles(pa, stream);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_chain_mu);
  ChainParams& P = g_chain_params;
  P = ChainParams();
  P.n = n;
  P.b = b;
  P.counter = a.counter;
  MapTable maps{&P};
  const long long rows = static_cast<long long>(n) * b;
  const int hi = maps.add(a.q_hi, rows, b);
  const int lo = maps.add(a.q_lo, rows, b);
  const int two = maps.add(a.two_i, b, b);
  int ph = 0;
  if (k == 3) {
    // R_3 = I + 2Q + Q^2 (2I + 2Q + Q^2): two dependent products instead of
    // three (the even/odd split of the Neumann polynomial in Q^2).
    //   phase 1: Q2 = Q_hi Q_hi
    //   phase 2: block = I + Q_hi 2I + Q_lo 2I + Q2 2I + (2 Q_hi) Q2 + Q2 Q2
    const int q2 = maps.add(a.e16[0], rows, b);
    const int hi2 = maps.add(a.e16[1], rows, b);  // 2 Q_hi from the prep launch
    ChainProd& P1 = P.phases[ph].prod[0];
    P.phases[ph++].nprod = 1;
    P1.nterms = 1;
    P1.term[0] = term(hi, hi, true);
    P1.mode = PROD_STORE;
    P1.epi = chain_epi(b);
    P1.epi.out_bf16 = a.e16[0];
    ChainProd& P2 = P.phases[ph].prod[0];
    P.phases[ph].lazy = 1;  // Q_hi 2I, Q_lo 2I need no phase-1 output
    P.phases[ph++].nprod = 1;
    P2.nterms = 5;
    P2.term[0] = term_2i(hi, two);
    P2.term[1] = term_2i(lo, two);
    P2.term[2] = dep_on(term_2i(q2, two), 0);
    P2.term[3] = dep_on(term(hi2, q2, true), 0);
    P2.term[4] = dep_on(term(q2, q2, true), 0);
    P2.mode = PROD_STORE;
    P2.epi = chain_epi(b);
    P2.epi.delta = 1.f;
    P2.epi.out_bf16 = a.blocks;
    P.nphases = ph;
    if (!maps.ok) return cudaErrorInvalidValue;
    return launch_chain(P, stream);
  }
  int cur = hi;  // E_{k+1} = Q
  __nv_bfloat16* ebuf[2] = {a.e16[0], a.e16[1]};
  int nxt = 0;
  for (int i = k; i >= 1; --i) {
    // E_i = Q E_{i+1} + 2Q,  2Q = Q_hi 2I + Q_lo 2I;  block = I + E_1
    ChainPhase& PH = P.phases[ph++];
    PH.nprod = 1;
    ChainProd& PR = PH.prod[0];
    PR.nterms = 3;
    PR.term[0] = term(hi, cur, true);
    PR.term[1] = term_2i(hi, two);
    PR.term[2] = term_2i(lo, two);
    PR.mode = PROD_STORE;
    EpiArgs ep = chain_epi(b);
    if (i == 1) {
      ep.delta = 1.f;
      ep.out_bf16 = a.blocks;
    } else {
      ep.out_bf16 = ebuf[nxt];
      cur = maps.add(ebuf[nxt], rows, b);
      nxt ^= 1;
    }
    PR.epi = ep;
  }
  P.nphases = ph;
  if (!maps.ok) return cudaErrorInvalidValue;
  return launch_chain(P, stream);
}

cudaError_t chain_adjoint(const ChainAdjointArgs& a, cudaStream_t stream) {
  const int k = a.k, b = a.b, n = a.n_a + a.n_b;
  if (!chain_fits(n, b, k)) return cudaErrorInvalidValue;
  PrepTilesArgs pa;  // Q (bf16), 2I, F_1 = G^T summed over the K splits
  pa.n_a = a.n_a;
  pa.n_b = a.n_b;
  pa.b = b;
  pa.theta_a = a.theta_a;
  pa.theta_b = a.theta_b;
  pa.q_hi = a.q16;
  pa.two_i = a.two_i;
  pa.part_a = a.part_a;
  pa.part_b = a.part_b;
  pa.splits_a = a.splits_a;
  pa.splits_b = a.splits_b;
  pa.nsb_a = a.nsb_a;
  pa.nsb_b = a.nsb_b;
  pa.S = a.S;
  pa.f16 = a.f16[0];
  pa.q_x2 = k == 3 ? a.x16 : nullptr;
  pa.zero_words = a.counter;
  pa.n_zero_words = kChainMaxPhases;
  if (k == 3 && a.x16 == nullptr) return cudaErrorInvalidValue;
  cudaError_t e = launch_prep_tiles(pa, stream);
  if (e != cudaSuccess) return e;
  if (k == 3) {
    // Adjoint of R = I + 2Q + Q2 M, M = 2I + 2Q + Q2, Q2 = Q Q, on transposes
    // (H = G^T, D = dQ^T), with Q^T = -Q and Q2^T = Q2:
    //   phase 1: Q2 = Q Q,  Q2d = (2Q) Q
    //   phase 2: D2 = dQ2^T = H 2I + (2Q) H + Q2 H + H Q2
    //   phase 3: D = H 2I + H Q2d + Q D2 + D2 Q
    // three dependent products instead of 2k - 1 = 5.
    std::lock_guard<std::mutex> lock(g_chain_mu);
    ChainParams& P = g_chain_params;
    P = ChainParams();
    P.n = n;
    P.b = b;
    P.counter = a.counter;
    MapTable maps{&P};
    const long long rows = static_cast<long long>(n) * b;
    const int q = maps.add(a.q16, rows, b);
    const int x = maps.add(a.x16, rows, b);
    const int two = maps.add(a.two_i, b, b);
    const int h = maps.add(a.f16[0], rows, b);
    const int q2 = maps.add(a.e16[2], rows, b);
    const int q2d = maps.add(a.e16[3], rows, b);
    const int d2 = maps.add(a.f16[1], rows, b);
    ChainPhase& P1 = P.phases[0];
    P1.nprod = 2;
    P1.prod[0].nterms = 1;
    P1.prod[0].term[0] = term(q, q, true);
    P1.prod[0].mode = PROD_STORE;
    P1.prod[0].epi = chain_epi(b);
    P1.prod[0].epi.out_bf16 = a.e16[2];
    P1.prod[1].nterms = 1;
    P1.prod[1].term[0] = term(x, q, true);
    P1.prod[1].mode = PROD_STORE;
    P1.prod[1].epi = chain_epi(b);
    P1.prod[1].epi.out_bf16 = a.e16[3];
    ChainProd& P2 = P.phases[1].prod[0];
    P.phases[1].nprod = 1;
    P.phases[1].lazy = 1;  // H 2I and (2Q) H need no phase-1 output
    P2.nterms = 4;
    P2.term[0] = term_2i(h, two);
    P2.term[1] = term(x, h, true);
    P2.term[2] = dep_on(term(q2, h, true), 0);
    P2.term[3] = dep_on(term(h, q2, true), 0);
    P2.mode = PROD_STORE;
    P2.epi = chain_epi(b);
    P2.epi.out_bf16 = a.f16[1];
    ChainProd& P3 = P.phases[2].prod[0];
    P.phases[2].nprod = 1;
    P.phases[2].lazy = 1;
    P3.nterms = 4;
    P3.term[0] = term_2i(h, two);
    P3.term[1] = dep_on(term(h, q2d, true), 0);
    P3.term[2] = dep_on(term(q, d2, true), 1);
    P3.term[3] = dep_on(term(d2, q, true), 1);
    P3.mode = PROD_STORE;
    P3.epi = chain_epi(b);
    P3.epi.out_f32 = a.d32;
    P.nphases = 3;
    if (!maps.ok) return cudaErrorInvalidValue;
    e = launch_chain(P, stream);
    if (e != cudaSuccess) return e;
  } else {
    std::lock_guard<std::mutex> lock(g_chain_mu);
    ChainParams& P = g_chain_params;
    P = ChainParams();
    P.n = n;
    P.b = b;
    P.counter = a.counter;
    MapTable maps{&P};
    const long long rows = static_cast<long long>(n) * b;
    const int q = maps.add(a.q16, rows, b);
    const int two = maps.add(a.two_i, b, b);
    int e_map[kChainMaxK + 2];
    e_map[k + 1] = q;
    int ph = 0;
    // E_i = Q E_{i+1} + Q 2I, i = k .. 2
    for (int i = k; i >= 2; --i) {
      ChainPhase& PH = P.phases[ph++];
      PH.nprod = 1;
      ChainProd& PR = PH.prod[0];
      PR.nterms = 2;
      PR.term[0] = term(q, e_map[i + 1], true);
      PR.term[1] = term_2i(q, two);
      PR.mode = PROD_STORE;
      EpiArgs ep = chain_epi(b);
      ep.out_bf16 = a.e16[i];
      PR.epi = ep;
      e_map[i] = maps.add(a.e16[i], rows, b);
    }
    // transposed reverse sweep with D = dQ^T in TMEM:
    //   i < k:  D += E_{i+1} F_i + F_i 2I,   F_{i+1} = F_i Q
    //   i = k:  D += Q F_k + F_k 2I + F_k Q   (the last term is F_{k+1})
    int cur = 0;
    for (int i = 1; i <= k; ++i) {
      ChainPhase& PH = P.phases[ph++];
      const int f = maps.add(a.f16[cur], rows, b);
      ChainProd& D = PH.prod[0];
      D.term[0] = term(e_map[i + 1], f, true);
      D.term[1] = term_2i(f, two);
      D.nterms = 2;
      D.first_acc = i == 1 ? 1 : 0;
      if (i < k) {
        D.mode = PROD_ACC;
        PH.nprod = 2;
        ChainProd& F = PH.prod[1];
        F.nterms = 1;
        F.term[0] = term(f, q, true);
        F.mode = PROD_STORE;
        EpiArgs ep = chain_epi(b);
        ep.out_bf16 = a.f16[1 - cur];
        F.epi = ep;
        cur = 1 - cur;
      } else {
        D.term[2] = term(f, q, true);
        D.nterms = 3;
        D.mode = PROD_ACC_STORE;
        EpiArgs ep = chain_epi(b);
        ep.out_f32 = a.d32;
        D.epi = ep;
        PH.nprod = 1;
      }
    }
    P.nphases = ph;
    if (!maps.ok) return cudaErrorInvalidValue;
    e = launch_chain(P, stream);
    if (e != cudaSuccess) return e;
  }
  // D = dQ^T: pack(dQ - dQ^T) = -pack(D - D^T)
  return launch_pack_tiles(a.d32, -1.f, a.n_a, a.n_b, b, a.dtheta_a, a.dtheta_b, stream);
}

}  // namespace poetx
