// C ABI of the POET-X layer (declared in include/poetx.h): argument checks,
// workspace carving, and the order of kernels for the block build, the
// forward and the backward pass.
//
// Dataflow (token-major rows; per token y_t = R (W0 (P x_t))):
//   build   : theta -> Q (unpack) -> E_{k+1} = Q, E_i = 2Q + Q E_{i+1}
//             -> block = I + E_1 = (I+Q)(I+Q+...+Q^k)
//   forward : u = x P^T (block-diagonal), v = u W0^T, y = v R^T
//   backward: dv = dy R, G_R = sum_t dy_t v_t^T, du = dv W0,
//             dx = du P, G_P = sum_t du_t x_t^T, then for each side the
//             reverse-mode sweep of the E recursion and the skew pack.
// bf16 mode runs every contraction on the tcgen05 engine; narrow blocks
// (b < 256) are placed on the diagonal of 256-wide zero-padded superblocks
// so the token-wise contractions always see 256 x 256 operands.  fp32 mode
// runs every contraction on the FFMA engine.
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "internal.h"
#include "poetx.h"

namespace poetx {

// ------------------------------------------------------------ bookkeeping

__device__ int g_status_word;

// Per-device caches below are filled on first use; several host threads may
// race to fill one, which is harmless (they store the same value).
int* device_status_ptr() {
  static std::atomic<int*> ptrs[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return nullptr;
  int* p = ptrs[dev].load(std::memory_order_relaxed);
  if (p == nullptr) {
    void* sym = nullptr;
    if (cudaGetSymbolAddress(&sym, g_status_word) == cudaSuccess) {
      p = static_cast<int*>(sym);
      ptrs[dev].store(p, std::memory_order_relaxed);
    }
  }
  return p;
}

int read_and_clear_device_status() {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof(int)) != cudaSuccess) return -1;
  const int zero = 0;
  cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int));
  return v;
}

int sm_count() {
  static std::atomic<int> counts[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 1;
  int n = counts[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    int c = 0;
    cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev);
    n = c > 0 ? c : 1;
    counts[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

namespace {

struct ProfRecord {
  const char* tag;
  cudaEvent_t start, stop;
  bool closed;
};

std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<cudaEvent_t> g_prof_pool;
std::vector<ProfRecord> g_prof_recs;
size_t g_prof_used = 0;
std::atomic<long long> g_launches{0};

}  // namespace

void prof_begin(const char* tag, cudaStream_t s) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (!g_prof_on || g_prof_used + 2 > g_prof_pool.size()) return;
  ProfRecord r{tag, g_prof_pool[g_prof_used], g_prof_pool[g_prof_used + 1], false};
  g_prof_used += 2;
  cudaEventRecord(r.start, s);
  g_prof_recs.push_back(r);
}

void prof_end(const char* tag, cudaStream_t s) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  if (g_prof_recs.empty()) return;
  ProfRecord& r = g_prof_recs.back();
  if (r.closed || std::strcmp(r.tag, tag) != 0) return;
  cudaEventRecord(r.stop, s);
  r.closed = true;
}

namespace {

using bf16 = __nv_bfloat16;

// ---------------------------------------------------------------- helpers

struct Carver {
  char* base;
  size_t off = 0;
  explicit Carver(void* b) : base(static_cast<char*>(b)) {}
  template <class T>
  T* take(size_t count) {
    off = (off + 255) & ~static_cast<size_t>(255);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += count * sizeof(T);
    return p;
  }
};

#define CK(expr)                                    \
  do {                                              \
    cudaError_t e_ = (expr);                        \
    if (e_ != cudaSuccess) return e_;               \
  } while (0)

constexpr long long kMaxTokens = 1ll << 22;
constexpr int kTargetCtas = 152;  // split-K sizing; fixed so results do not depend on the device

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

poetx_status check_dims(int d, int b, bool is_bf16) {
  if (b < 2 || b > 512 || d <= 0 || d % b != 0) return POETX_ERR_INVALID_ARG;
  if (static_cast<long long>(d) * b > (1ll << 30)) return POETX_ERR_UNSUPPORTED;
  if (is_bf16) {
    if (b != 32 && b != 64 && b != 128 && b != 256 && b != 512) return POETX_ERR_UNSUPPORTED;
    const int S = b > 256 ? b : 256;
    if (d % S != 0) return POETX_ERR_UNSUPPORTED;
  }
  return POETX_OK;
}

poetx_status check_common(int b, int k, long long tokens, poetx_dtype dtype) {
  if (dtype != POETX_F32 && dtype != POETX_BF16) return POETX_ERR_INVALID_ARG;
  if (k < 0 || k > 16) return POETX_ERR_INVALID_ARG;
  if (tokens < 0 || tokens > kMaxTokens) return POETX_ERR_INVALID_ARG;
  (void)b;
  return POETX_OK;
}

poetx_status to_status(cudaError_t e) { return e == cudaSuccess ? POETX_OK : POETX_ERR_CUDA; }

int superblock(int b) { return b > 256 ? b : 256; }
bool tc_small(bool is_bf16, int b) { return is_bf16 && b >= 128; }

// The b x b chains run as one cooperative launch each where they fit
// (chain_tc.cu); otherwise as one launch per product.
constexpr bool kChainEnabled = true;

bool use_chain(bool is_bf16, int n, int b, int k) {
  return kChainEnabled && tc_small(is_bf16, b) && chain_fits(n, b, k);
}

TcOperand op(const void* ptr, long long rows, long long cols, long long pitch, bool mn_major,
             int mn_per_g, int k_per_g) {
  TcOperand o;
  o.ptr = ptr;
  o.rows = rows;
  o.cols = cols;
  o.pitch = pitch;
  o.mn_major = mn_major;
  o.mn_per_g = mn_per_g;
  o.k_per_g = k_per_g;
  return o;
}

int outer_splits(int d, int S, long long T) {
  const int tiles = (d / S) * (S / 128) * (S / 256);
  int splits = kTargetCtas / (tiles > 0 ? tiles : 1);
  const long long ksteps = (T + 63) / 64;
  long long cap = ksteps / 4;
  if (cap < 1) cap = 1;
  if (splits > cap) splits = static_cast<int>(cap);
  if (splits < 1) splits = 1;
  return tc_effective_splits(static_cast<int>(T), splits);
}

// ------------------------------------------------- token-wise contractions

// out[:, sb g] = in[:, sb g] * SB_g^T (or * SB_g when transposed), bf16.
cudaError_t tc_transform(const bf16* in, const bf16* sb, bf16* out, int d, int S, long long T,
                         bool transposed, const char* tag, cudaStream_t s) {
  TcGemm g;
  g.M = static_cast<int>(T);
  g.N = S;
  g.K = S;
  g.batches = d / S;
  // S = 256: the block (256 x 256 bf16, 128 KiB) stays resident while a CTA
  // walks token tiles; S = 512: 256-wide tiles with the block's rows streamed
  // (a resident 512 x 128 slice gives N = 128 tiles whose K steps hold too
  // little MMA work to cover the loads)
  g.BN = 256;
  g.b_resident = S == 256;
  g.A = op(in, T, d, d, false, 0, S);
  g.B = transposed ? op(sb, d, S, S, true, 0, S) : op(sb, d, S, S, false, S, 0);
  g.epi.out_bf16 = out;
  g.epi.ld = d;
  g.epi.col_g = S;
  g.epi.row_limit = static_cast<int>(T);
  g.epi.out_rows = T;
  g.tag = tag;
  return tc_gemm_run(g, s);
}

// part[s][g][m][n] = sum over tokens of split s of A[t][g*S+m] * B[t][g*S+n].
cudaError_t tc_outer(const bf16* A, const bf16* B, float* part, int d, int S, long long T,
                     int splits, cudaStream_t s) {
  TcGemm g;
  g.M = S;
  g.N = S;
  g.K = static_cast<int>(T);
  g.batches = d / S;
  g.splits = splits;
  g.BN = 256;
  g.A = op(A, T, d, d, true, S, 0);
  g.B = op(B, T, d, d, true, S, 0);
  g.epi.out_f32 = part;
  g.epi.ld = S;
  g.epi.row_g = S;
  g.epi.row_s = (d / S) * S;
  g.epi.out_rows = static_cast<long long>(splits) * (d / S) * S;
  g.tag = "outer";
  return tc_gemm_run(g, s);
}

// The W0 GEMMs run as clusters of two CTAs that share each B (W0) tile.
constexpr bool kW0Clusters = true;

// The last, partial round of W0 GEMM tiles is spread one tile per cluster
// with its K steps split between the two CTAs (poetx_set_w0_split_tail).
std::atomic<int> g_w0_split_tail{1};

// The W0 GEMMs run on CTA pairs (one 256-row MMA per K slice across two
// SMs); off: clusters of two one-CTA MMAs (poetx_set_w0_pair_mma).
std::atomic<int> g_w0_pair{1};

// v = u W0^T (fwd) or du = dv W0 (dgrad), bf16.
cudaError_t tc_w0(const bf16* A, const bf16* W0, bf16* out, int d_in, int d_out, long long T,
                  bool dgrad, cudaStream_t s) {
  TcGemm g;
  g.M = static_cast<int>(T);
  g.BN = 256;
  if (!dgrad) {
    g.N = d_out;
    g.K = d_in;
    g.A = op(A, T, d_in, d_in, false, 0, 0);
    g.B = op(W0, d_out, d_in, d_in, false, 0, 0);
    g.epi.ld = d_out;
    g.tag = "gemm_w0";
  } else {
    g.N = d_in;
    g.K = d_out;
    g.A = op(A, T, d_out, d_out, false, 0, 0);
    g.B = op(W0, d_out, d_in, d_in, true, 0, 0);
    g.epi.ld = d_in;
    g.tag = "gemm_w0_dgrad";
  }
  g.epi.out_bf16 = out;
  g.epi.row_limit = static_cast<int>(T);
  g.epi.out_rows = T;
  g.cluster2 = kW0Clusters;
  g.split_tail = g_w0_split_tail.load(std::memory_order_relaxed) != 0;
  if (g_w0_pair.load(std::memory_order_relaxed) != 0) return w0_pair_run(g, s);
  return tc_gemm_run(g, s);
}

// The W0 GEMMs with the block-diagonal factor applied in the epilogue (256 x
// 256 superblocks): fwd v = u W0^T and y = v R^T per block; dgrad du = dv W0
// and dx = du P per block.  `out` (v or du) may be null: then only the
// block output is written.  Off unless poetx_set_block_epilogue_fusion(1):
// its 64 KiB staging tile leaves a 3-stage operand ring, and the GEMM then
// loses more than the separate block transform costs.
std::atomic<int> g_fuse_block_epilogue{0};

bool fuse_block_epilogue(bool is_bf16, int b) {
  return g_fuse_block_epilogue.load(std::memory_order_relaxed) != 0 && is_bf16 && b <= 256;
}

cudaError_t tc_w0_block(const bf16* A, const bf16* W0, const bf16* sb, bf16* out, bf16* out_blk,
                        int d_in, int d_out, long long T, bool dgrad, cudaStream_t s) {
  TcGemm g;
  g.M = static_cast<int>(T);
  g.BN = 256;
  if (!dgrad) {
    g.N = d_out;
    g.K = d_in;
    g.A = op(A, T, d_in, d_in, false, 0, 0);
    g.B = op(W0, d_out, d_in, d_in, false, 0, 0);
    g.blk = op(sb, d_out, 256, 256, false, 0, 0);  // blk_j[n][kk] = R_j[n][kk]
    g.epi.ld = d_out;
    g.tag = "gemm_w0_r";
  } else {
    g.N = d_in;
    g.K = d_out;
    g.A = op(A, T, d_out, d_out, false, 0, 0);
    g.B = op(W0, d_out, d_in, d_in, true, 0, 0);
    g.blk = op(sb, d_in, 256, 256, true, 0, 0);  // rows kk, columns n of P_j
    g.epi.ld = d_in;
    g.tag = "gemm_w0_dgrad_p";
  }
  g.epi.out_bf16 = out;
  g.out_blk = out_blk;
  g.epi.row_limit = static_cast<int>(T);
  g.epi.out_rows = T;
  if (g_w0_pair.load(std::memory_order_relaxed) != 0) return w0_pair_run(g, s);
  return tc_gemm_run(g, s);
}

// fp32 block-diagonal transform: out[:, g] = in[:, g] B_g^T (or B_g).
cudaError_t simt_transform(const float* in, const float* blocks, float* out, int d, int b,
                           long long T, bool transposed, const char* tag, cudaStream_t s) {
  SimtGemm g;
  g.M = static_cast<int>(T);
  g.N = b;
  g.K = b;
  g.batches = d / b;
  g.A = in;
  g.a_g = b;
  g.a_m = d;
  g.a_k = 1;
  g.B = blocks;
  g.b_g = static_cast<long long>(b) * b;
  if (!transposed) {  // B(kk=j, n=i) = B_g[i][j]
    g.b_k = 1;
    g.b_n = b;
  } else {  // B(kk=j, n=i) = B_g[j][i]
    g.b_k = b;
    g.b_n = 1;
  }
  g.epi.out_f32 = out;
  g.epi.ld = d;
  g.epi.col_g = b;
  g.tag = tag;
  return simt_gemm_run(g, s);
}

// fp32 G[g][i][j] = sum_t A[t][g*b+i] B[t][g*b+j].
cudaError_t simt_outer(const float* A, const float* B, float* G, int d, int b, long long T,
                       cudaStream_t s) {
  SimtGemm g;
  g.M = b;
  g.N = b;
  g.K = static_cast<int>(T);
  g.batches = d / b;
  g.A = A;
  g.a_g = b;
  g.a_m = 1;
  g.a_k = d;
  g.B = B;
  g.b_g = b;
  g.b_k = d;
  g.b_n = 1;
  g.epi.out_f32 = G;
  g.epi.ld = b;
  g.epi.row_g = b;
  g.tag = "outer";
  return simt_gemm_run(g, s);
}

cudaError_t simt_w0(const float* A, const float* W0, float* out, int d_in, int d_out,
                    long long T, bool dgrad, cudaStream_t s) {
  SimtGemm g;
  g.M = static_cast<int>(T);
  g.batches = 1;
  g.A = A;
  g.a_k = 1;
  g.B = W0;
  if (!dgrad) {  // v[t][o] = sum_i u[t][i] W0[o][i]
    g.N = d_out;
    g.K = d_in;
    g.a_m = d_in;
    g.b_k = 1;
    g.b_n = d_in;
    g.epi.ld = d_out;
    g.tag = "gemm_w0";
  } else {  // du[t][i] = sum_o dv[t][o] W0[o][i]
    g.N = d_in;
    g.K = d_out;
    g.a_m = d_out;
    g.b_k = d_in;
    g.b_n = 1;
    g.epi.ld = d_in;
    g.tag = "gemm_w0_dgrad";
  }
  g.epi.out_f32 = out;
  return simt_gemm_run(g, s);
}

// ------------------------------------------------------- b x b products

// out = epi(L * Rm) over n blocks, where L = Q (or Q^T) and Rm = one of the
// E / G matrices, chosen by `kind`:
//   kind 0: Q * M          (builder recursion E_i = 2Q + Q E_{i+1})
//   kind 1: M * N^T        (adjoint: G_i E_{i+1}^T)
//   kind 2: Q^T * M        (adjoint: G_{i+1} = Q^T G_i)
// tc: operands bf16 (q16 / m16 / n16); otherwise fp32 (q32 / m32 / n32).
cudaError_t small_product(int kind, bool tc, int n, int b, const float* q32, const bf16* q16,
                          const float* m32, const bf16* m16, const float* n32, const bf16* n16,
                          const EpiArgs& epi, const char* tag, cudaStream_t s) {
  const long long bb = static_cast<long long>(b) * b;
  const long long rows = static_cast<long long>(n) * b;
  if (tc) {
    TcGemm g;
    g.M = b;
    g.N = b;
    g.K = b;
    g.batches = n;
    g.BN = 128;  // b >= 128 here; 128-wide tiles give twice the CTAs of 256-wide ones
    if (kind == 0) {
      g.A = op(q16, rows, b, b, false, b, 0);  // A[m][kk] = Q[m][kk]
      g.B = op(m16, rows, b, b, true, 0, b);   // B[nn][kk] = M[kk][nn]
    } else if (kind == 1) {
      g.A = op(m16, rows, b, b, false, b, 0);  // A[m][kk] = M[m][kk]
      g.B = op(n16, rows, b, b, false, b, 0);  // B[nn][kk] = N[nn][kk]
    } else {
      g.A = op(q16, rows, b, b, true, 0, b);   // A[m][kk] = Q[kk][m]
      g.B = op(m16, rows, b, b, true, 0, b);   // B[nn][kk] = M[kk][nn]
    }
    g.epi = epi;
    g.tag = tag;
    return tc_gemm_run(g, s);
  }
  SimtGemm g;
  g.M = b;
  g.N = b;
  g.K = b;
  g.batches = n;
  g.a_g = bb;
  g.b_g = bb;
  if (kind == 0) {
    g.A = q32;
    g.a_m = b;
    g.a_k = 1;
    g.B = m32;
    g.b_k = b;
    g.b_n = 1;
  } else if (kind == 1) {
    g.A = m32;
    g.a_m = b;
    g.a_k = 1;
    g.B = n32;
    g.b_k = 1;
    g.b_n = b;
  } else {
    g.A = q32;
    g.a_m = 1;
    g.a_k = b;
    g.B = m32;
    g.b_k = b;
    g.b_n = 1;
  }
  g.epi = epi;
  g.tag = tag;
  return simt_gemm_run(g, s);
}

EpiArgs block_epi(int b) {  // [n][b][b] row-major outputs and addends
  EpiArgs e;
  e.ld = b;
  e.row_g = b;
  return e;
}

// --------------------------------------------------------------- builder

struct BuildBufs {
  float* q32 = nullptr;
  bf16* q16 = nullptr;
  float* e32[2] = {nullptr, nullptr};
  bf16* e16[2] = {nullptr, nullptr};
  unsigned int* counter = nullptr;  // grid barrier of the chain launch
  bf16* q_lo = nullptr;             // chain: bf16 remainder Q - bf16(Q)
  bf16* two_i = nullptr;            // chain: constant 2I
};

// Buffers of one block build: the one-launch chain needs bf16 Q (hi and lo
// parts), 2I and two bf16 E stacks; the per-product path fp32 Q plus bf16 (tensor
// cores) or fp32 (FFMA) E stacks.
// The build of bf16 blocks with b <= 256 and 1 <= k <= 16 runs on CTA pairs
// with its operands in shared memory (cnp_pair.cu): no workspace.
bool use_pair_build(bool is_bf16, int n, int b, int k) {
  return is_bf16 && cnp_pair_fits(b, k) && (static_cast<long long>(n) * b) % 256 == 0;
}

BuildBufs carve_build(Carver& c, int n, int b, int k, bool is_bf16) {
  BuildBufs w;
  if (use_pair_build(is_bf16, n, b, k)) return w;
  const size_t nbb = static_cast<size_t>(n) * b * b;
  if (use_chain(is_bf16, n, b, k)) {
    w.q16 = c.take<bf16>(nbb);
    w.q_lo = c.take<bf16>(nbb);
    w.e16[0] = c.take<bf16>(nbb);
    w.e16[1] = c.take<bf16>(nbb);
    w.two_i = c.take<bf16>(static_cast<size_t>(b) * b);
    w.counter = c.take<unsigned int>(kChainMaxPhases);
    return w;
  }
  w.q32 = c.take<float>(nbb);
  if (tc_small(is_bf16, b)) {
    w.q16 = c.take<bf16>(nbb);
    w.e16[0] = c.take<bf16>(nbb);
    w.e16[1] = c.take<bf16>(nbb);
  } else {
    w.e32[0] = c.take<float>(nbb);
    w.e32[1] = c.take<float>(nbb);
  }
  return w;
}

cudaError_t run_build(const float* theta, int n, int b, int k, bool is_bf16, void* blocks,
                      const BuildBufs& w, cudaStream_t s) {
  const bool tc = tc_small(is_bf16, b);
  if (use_pair_build(is_bf16, n, b, k))
    return cnp_build_pair(theta, n, b, k, static_cast<bf16*>(blocks), s);
  if (use_chain(is_bf16, n, b, k)) {  // the whole recursion in one cooperative launch
    ChainBuildArgs a;
    a.n = n;
    a.b = b;
    a.k = k;
    a.theta = theta;
    a.q_hi = w.q16;
    a.q_lo = w.q_lo;
    a.two_i = w.two_i;
    a.e16[0] = w.e16[0];
    a.e16[1] = w.e16[1];
    a.counter = w.counter;
    a.blocks = static_cast<bf16*>(blocks);
    return chain_build(a, s);
  }
  float* out32 = is_bf16 ? nullptr : static_cast<float*>(blocks);
  bf16* out16 = is_bf16 ? static_cast<bf16*>(blocks) : nullptr;
  if (!tc && small_chain_fits(b))  // the whole recursion per block in one CTA
    return launch_small_build(theta, n, b, k, out32, out16, s);
  CK(launch_unpack(theta, n, nullptr, 0, b, w.q32, tc ? w.q16 : nullptr, s));
  if (k == 0) return launch_identity_plus(w.q32, n, b, out32, out16, s);
  int cur = -1;  // -1: E_{k+1} = Q itself
  for (int i = k; i >= 1; --i) {
    const int nxt = cur == 0 ? 1 : 0;
    EpiArgs e = block_epi(b);
    e.X = w.q32;  // + 2 Q
    e.beta = 2.f;
    if (i == 1) {
      e.delta = 1.f;  // + I
      e.out_f32 = out32;
      e.out_bf16 = out16;
    } else if (tc) {
      e.out_bf16 = w.e16[nxt];
    } else {
      e.out_f32 = w.e32[nxt];
    }
    const float* m32 = cur < 0 ? w.q32 : w.e32[cur];
    const bf16* m16 = cur < 0 ? w.q16 : w.e16[cur];
    CK(small_product(0, tc, n, b, w.q32, w.q16, m32, m16, nullptr, nullptr, e, "build", s));
    cur = nxt;
  }
  return cudaSuccess;
}

// -------------------------------------------------- adjoint of the build

struct CnpBufs {
  float* q32 = nullptr;
  bf16* q16 = nullptr;
  float* e32[18] = {};
  bf16* e16[18] = {};
  float* g32[2] = {nullptr, nullptr};
  bf16* g16[2] = {nullptr, nullptr};
  float* dq = nullptr;
  unsigned int* counter = nullptr;
  bf16* two_i = nullptr;  // chain: constant 2I
  bf16* x16 = nullptr;    // chain, k = 3: 2Q
  // the adjoint on CTA pairs (1 <= k <= 16, b <= 256): H (bf16) per
  // 256 x 256 superblock
  bool pair = false;
  bf16* hg = nullptr;
};

CnpBufs carve_cnp(Carver& c, int n, int b, int k, bool is_bf16) {
  CnpBufs w;
  if (use_pair_build(is_bf16, n, b, k)) {
    const size_t sq = static_cast<size_t>(n) * b * 256;  // superblocks x 256 x 256
    w.pair = true;
    w.hg = c.take<bf16>(sq);
    return w;
  }
  const bool tc = tc_small(is_bf16, b);
  const size_t nbb = static_cast<size_t>(n) * b * b;
  w.q32 = c.take<float>(nbb);
  if (tc) w.q16 = c.take<bf16>(nbb);
  for (int i = 2; i <= k; ++i) {
    if (tc)
      w.e16[i] = c.take<bf16>(nbb);
    else
      w.e32[i] = c.take<float>(nbb);
  }
  for (int j = 0; j < 2; ++j) {
    w.g32[j] = c.take<float>(nbb);
    if (tc) w.g16[j] = c.take<bf16>(nbb);
  }
  w.dq = c.take<float>(nbb);
  if (tc) {
    w.counter = c.take<unsigned int>(kChainMaxPhases);
    w.two_i = c.take<bf16>(static_cast<size_t>(b) * b);
    if (k == 3) w.x16 = c.take<bf16>(nbb);
  }
  return w;
}



// The adjoint (on CTA pairs, else the one-launch chain) for blocks [0, n_a)
// (side a) and [n_a, n_a + n_b) (side b)
// from the split-K partials of the transposed block gradients.
cudaError_t chain_adjoint_from_parts(const float* theta_a, int n_a, const float* part_a,
                                     int splits_a, const float* theta_b, int n_b,
                                     const float* part_b, int splits_b, int b, int k,
                                     const CnpBufs& w, float* dtheta_a, float* dtheta_b,
                                     cudaStream_t s) {
  if (w.pair) {  // one launch on CTA pairs, superblocks of both sides
    CnpAdjointPairArgs x;
    x.n_a = n_a;
    x.n_b = n_b;
    x.b = b;
    x.k = k;
    x.theta_a = theta_a;
    x.theta_b = theta_b;
    x.part_a = part_a;
    x.part_b = part_b;
    x.splits_a = splits_a;
    x.splits_b = splits_b;
    x.hg = w.hg;
    x.dtheta_a = dtheta_a;
    x.dtheta_b = dtheta_b;
    return cnp_adjoint_pair(x, s);
  }
  ChainAdjointArgs a;
  a.n_a = n_a;
  a.n_b = n_b;
  a.b = b;
  a.k = k;
  a.theta_a = theta_a;
  a.theta_b = theta_b;
  a.q16 = w.q16;
  a.two_i = w.two_i;
  for (int i = 2; i <= k; ++i) a.e16[i] = w.e16[i];
  a.f16[0] = w.g16[0];
  a.f16[1] = w.g16[1];
  a.x16 = w.x16;
  a.d32 = w.dq;
  a.S = superblock(b);
  a.part_a = part_a;
  a.splits_a = splits_a;
  a.nsb_a = n_a * b / a.S;
  a.part_b = part_b;
  a.splits_b = splits_b;
  a.nsb_b = n_b * b / a.S;
  a.dtheta_a = dtheta_a;
  a.dtheta_b = dtheta_b;
  a.counter = w.counter;
  return chain_adjoint(a, s);
}

// Input: the block gradients G of n = n_a + n_b blocks in w.g32[0] (and
// w.g16[0] for tc); blocks [0, n_a) belong to theta_a, the rest to theta_b.
// Reverse sweep of E_{k+1} = Q, E_i = c_i Q + Q E_{i+1} (c_i = 2), R = I + E_1:
//   Gbar_1 = G;  for i = 1..k:  dQ += 2 Gbar_i + Gbar_i E_{i+1}^T,
//                               Gbar_{i+1} = Q^T Gbar_i;
//   dQ += Gbar_{k+1};  dtheta = pack(dQ - dQ^T).
cudaError_t run_cnp_backward(const float* theta_a, int n_a, const float* theta_b, int n_b, int b,
                             int k, bool is_bf16, const CnpBufs& w, float* dtheta_a,
                             float* dtheta_b, cudaStream_t s) {
  const bool tc = tc_small(is_bf16, b);
  const int n = n_a + n_b;
  if (!tc && small_chain_fits(b))  // the whole adjoint per block in one CTA
    return launch_small_adjoint(theta_a, n_a, theta_b, n_b, b, k, w.g32[0], dtheta_a, dtheta_b,
                                s);
  if (k == 0) return launch_pack_skew(w.g32[0], nullptr, n_a, n_b, b, dtheta_a, dtheta_b, s);
  CK(launch_unpack(theta_a, n_a, theta_b, n_b, b, w.q32, tc ? w.q16 : nullptr, s));
  // E_i for i = k .. 2 (E_{k+1} = Q)
  for (int i = k; i >= 2; --i) {
    EpiArgs e = block_epi(b);
    e.X = w.q32;
    e.beta = 2.f;
    if (tc)
      e.out_bf16 = w.e16[i];
    else
      e.out_f32 = w.e32[i];
    const float* m32 = (i + 1 == k + 1) ? w.q32 : w.e32[i + 1];
    const bf16* m16 = (i + 1 == k + 1) ? w.q16 : w.e16[i + 1];
    CK(small_product(0, tc, n, b, w.q32, w.q16, m32, m16, nullptr, nullptr, e, "cnp_bwd", s));
  }
  int cur = 0;
  for (int i = 1; i <= k; ++i) {
    const float* e32 = (i + 1 == k + 1) ? w.q32 : w.e32[i + 1];
    const bf16* e16 = (i + 1 == k + 1) ? w.q16 : w.e16[i + 1];
    EpiArgs e1 = block_epi(b);
    if (i > 1) {
      e1.X = w.dq;
      e1.beta = 1.f;
    }
    e1.Y = w.g32[cur];
    e1.gamma = 2.f;
    e1.out_f32 = w.dq;
    CK(small_product(1, tc, n, b, nullptr, nullptr, w.g32[cur], w.g16[cur], e32, e16, e1,
                     "cnp_bwd", s));
    EpiArgs e2 = block_epi(b);
    e2.out_f32 = w.g32[1 - cur];
    if (tc) e2.out_bf16 = w.g16[1 - cur];
    CK(small_product(2, tc, n, b, w.q32, w.q16, w.g32[cur], w.g16[cur], nullptr, nullptr, e2,
                     "cnp_bwd", s));
    cur = 1 - cur;
  }
  return launch_pack_skew(w.dq, w.g32[cur], n_a, n_b, b, dtheta_a, dtheta_b, s);
}

// -------------------------------------------------------- layer buffers

struct SideBufs {  // token-wise scratch for one call
  void* u = nullptr;
  void* v = nullptr;
  void* dv = nullptr;
  void* du = nullptr;
  bf16* psb = nullptr;
  bf16* rsb = nullptr;
  float* part = nullptr;
};

size_t elem_size(bool is_bf16) { return is_bf16 ? 2 : 4; }

void* take_act(Carver& c, long long T, int d, bool is_bf16) {
  return c.take<char>(static_cast<size_t>(T) * d * elem_size(is_bf16));
}

struct FwdPlan {
  SideBufs sb;
};

FwdPlan carve_forward(Carver& c, int d_in, int d_out, int b, long long T, bool is_bf16,
                      bool need_v) {
  FwdPlan p;
  p.sb.u = take_act(c, T, d_in, is_bf16);
  if (need_v) p.sb.v = take_act(c, T, d_out, is_bf16);  // (unused by the fused forward)
  if (is_bf16 && b < 256) {
    p.sb.psb = c.take<bf16>(static_cast<size_t>(d_in) * 256);
    p.sb.rsb = c.take<bf16>(static_cast<size_t>(d_out) * 256);
  }
  return p;
}

cudaError_t run_forward_uv(const void* x, const void* W0, const void* psb, void* u, void* v,
                           int d_in, int d_out, int b, long long T, bool is_bf16,
                           cudaStream_t s) {
  if (is_bf16) {
    const int S = superblock(b);
    CK(tc_transform(static_cast<const bf16*>(x), static_cast<const bf16*>(psb),
                    static_cast<bf16*>(u), d_in, S, T, false, "transform", s));
    return tc_w0(static_cast<const bf16*>(u), static_cast<const bf16*>(W0), static_cast<bf16*>(v),
                 d_in, d_out, T, false, s);
  }
  CK(simt_transform(static_cast<const float*>(x), static_cast<const float*>(psb),
                    static_cast<float*>(u), d_in, b, T, false, "transform", s));
  return simt_w0(static_cast<const float*>(u), static_cast<const float*>(W0),
                 static_cast<float*>(v), d_in, d_out, T, false, s);
}

struct BwdPlan {
  SideBufs sb;
  CnpBufs cnp;
  float* part_out = nullptr;  // chain mode: the R side's partials live until the chain
  int splits_in = 1, splits_out = 1;
};

// The backward's transposed transforms and token sums run fused (one pass over
// dy and one over du) wherever the adjoint reads split-K partials of 256 x 256
// superblocks: the CTA-pair kernels and the one-launch chain up to b = 256.
bool use_transform_sum(bool is_bf16, int n, int b, int k) {
  return (use_chain(is_bf16, n, b, k) && b <= 256) || use_pair_build(is_bf16, n, b, k);
}

BwdPlan carve_backward(Carver& c, int d_in, int d_out, int b, int k, long long T, bool is_bf16,
                       bool recompute_v, bool fused) {
  BwdPlan p;
  if (recompute_v) {
    p.sb.u = take_act(c, T, d_in, is_bf16);
    p.sb.v = take_act(c, T, d_out, is_bf16);
  }
  p.sb.dv = take_act(c, T, d_out, is_bf16);
  p.sb.du = take_act(c, T, d_in, is_bf16);
  if (is_bf16) {
    const int S = superblock(b);
    if (b < 256) {
      p.sb.psb = c.take<bf16>(static_cast<size_t>(d_in) * 256);
      p.sb.rsb = c.take<bf16>(static_cast<size_t>(d_out) * 256);
    }
    const bool ts = use_transform_sum(is_bf16, (d_in + d_out) / b, b, k);
    // with the block factor in the dgrad GEMM's epilogue, G_P's token sums
    // run on their own (outer splits)
    p.splits_in = ts && !fused ? transform_sum_splits(d_in, T) : outer_splits(d_in, S, T);
    p.splits_out = ts ? transform_sum_splits(d_out, T) : outer_splits(d_out, S, T);
    const long long part_in = static_cast<long long>(p.splits_in) * d_in * S;
    const long long part_out = static_cast<long long>(p.splits_out) * d_out * S;
    if (use_chain(is_bf16, (d_in + d_out) / b, b, k) ||
        use_pair_build(is_bf16, (d_in + d_out) / b, b, k)) {  // both live until the adjoint
      p.sb.part = c.take<float>(static_cast<size_t>(part_in));
      p.part_out = c.take<float>(static_cast<size_t>(part_out));
    } else {
      p.sb.part = c.take<float>(static_cast<size_t>(part_in > part_out ? part_in : part_out));
    }
  }
  p.cnp = carve_cnp(c, (d_in + d_out) / b, b, k, is_bf16);
  return p;
}

// Block gradients G[g] = sum_t dout[t][g-block]^T in[t][g-block] of one side
// into g32 (+ g16 for the bf16 adjoint), [d/b][b][b].
cudaError_t block_gradient(const void* dout, const void* in, int d, int b, long long T,
                           bool is_bf16, float* part, int splits, float* g32, bf16* g16,
                           cudaStream_t s) {
  const int n = d / b;
  if (is_bf16) {
    const int S = superblock(b);
    CK(tc_outer(static_cast<const bf16*>(dout), static_cast<const bf16*>(in), part, d, S, T,
                splits, s));
    return launch_reduce_extract(part, splits, n, b, S, g32, tc_small(true, b) ? g16 : nullptr,
                                 s);
  }
  if (small_chain_fits(b))  // small blocks: one cluster per block
    return launch_small_outer(static_cast<const float*>(dout), static_cast<const float*>(in), g32,
                              d, b, T, s);
  return simt_outer(static_cast<const float*>(dout), static_cast<const float*>(in), g32, d, b, T,
                    s);
}

const void* superblocks_or_blocks(const void* blocks, bf16* sb, int d, int b, bool is_bf16,
                                  cudaStream_t s, cudaError_t* err) {
  *err = cudaSuccess;
  if (!is_bf16 || b >= 256) return blocks;
  *err = launch_expand_superblocks(static_cast<const bf16*>(blocks), d / b, b, 256, sb, s);
  return sb;
}

}  // namespace
}  // namespace poetx


// ===================================================== block build, no alloc
//
// Some callers cannot allocate device memory at the point where they need
// the block build: code running under an allocator that forbids new
// allocations (a static memory plan, a real-time loop, or an embedding
// framework that owns every device buffer and hands out only the tensors
// it planned), or a caller that simply has no workspace to offer.  For them
// poetx_build_blocks_noalloc runs the same kernels as poetx_build_blocks
// but takes its scratch from one file-scope device array of fixed size,
// created when the library's module is loaded on a GPU and held by every
// GPU that loads the library until the process exits.
//
// Host code may not use that array's name as a device address (in host
// code it names a host-side stand-in), so the device address is looked up
// with cudaGetSymbolAddress, with the device current, on every call made
// outside stream capture (the lookup follows the module if the context was
// destroyed and re-created, e.g. by cudaDeviceReset), and handed to the
// kernels.  A call made while its stream is being captured uses the address
// found by the last call outside capture on that device, so the first call
// on a device, and the first after a device reset, must come before any
// stream capture.
//
// Every call shares the one array and the array keeps whatever the last call
// left in it.  The build needs no part of it to start at zero: every word a
// call reads was written earlier in the same call.  Calls that overlap on
// the GPU (different streams, or different host threads, on one device)
// race on the array and must be serialised by the caller.

namespace poetx {
namespace {

// Largest build served: (d/b) * b * b = d * b <= 2^20 elements, e.g. d = 4096
// with b = 256, d = 2048 with b = 512 or d = 8192 with b = 128.  At that size
// the fp32 path needs three fp32 b x b stacks (12 MiB) and the bf16
// tensor-core path one fp32 and three bf16 stacks (10 MiB).
constexpr long long kNoAllocMaxElems = 1ll << 20;
constexpr size_t kNoAllocScratchBytes = (12u << 20) + 1024;

static __device__ __align__(256) unsigned char g_build_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;

// Device address of g_build_scratch on the current device (nullptr on
// failure): looked up when `stream` is not capturing, else the address the
// last lookup on this device found.
void* build_scratch_address(cudaStream_t stream) {
  static std::vector<void*> addr;  // by device ordinal
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return nullptr;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (static_cast<size_t>(dev) >= addr.size()) addr.resize(dev + 1, nullptr);
  if (cs == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_build_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace
}  // namespace poetx

using namespace poetx;

// ====================================================================== ABI

extern "C" {

const char* poetx_status_string(poetx_status s) {
  switch (s) {
    case POETX_OK: return "POETX_OK";
    case POETX_ERR_INVALID_ARG: return "POETX_ERR_INVALID_ARG: invalid argument";
    case POETX_ERR_UNSUPPORTED: return "POETX_ERR_UNSUPPORTED: shape not supported";
    case POETX_ERR_WORKSPACE: return "POETX_ERR_WORKSPACE: workspace too small";
    case POETX_ERR_CUDA: return "POETX_ERR_CUDA: CUDA launch or device error";
    case POETX_ERR_TIMEOUT: return "POETX_ERR_TIMEOUT: a kernel gave up on an internal wait";
  }
  return "unknown poetx_status";
}

size_t poetx_packed_size(int d, int b) {
  if (b < 1 || d <= 0 || d % b != 0) return 0;
  return static_cast<size_t>(d / b) * (static_cast<size_t>(b) * (b - 1) / 2);
}

size_t poetx_build_workspace_size(int d, int b, int k, poetx_dtype dtype) {
  const bool is_bf16 = dtype == POETX_BF16;
  if (check_dims(d, b, is_bf16) != POETX_OK || check_common(b, k, 0, dtype) != POETX_OK) return 0;
  Carver c(nullptr);
  carve_build(c, d / b, b, k, is_bf16);
  return c.off;
}

poetx_status poetx_build_blocks(const float* theta, int d, int b, int k, poetx_dtype dtype,
                                void* blocks, void* workspace, size_t workspace_bytes,
                                poetx_stream stream) {
  const bool is_bf16 = dtype == POETX_BF16;
  poetx_status st = check_common(b, k, 0, dtype);
  if (st != POETX_OK) return st;
  if ((st = check_dims(d, b, is_bf16)) != POETX_OK) return st;
  if (theta == nullptr || blocks == nullptr || !aligned16(theta) || !aligned16(blocks))
    return POETX_ERR_INVALID_ARG;
  Carver c(workspace);
  BuildBufs w = carve_build(c, d / b, b, k, is_bf16);
  if (c.off > 0 && (workspace == nullptr || c.off > workspace_bytes || !aligned16(workspace)))
    return POETX_ERR_WORKSPACE;
  return to_status(
      run_build(theta, d / b, b, k, is_bf16, blocks, w, static_cast<cudaStream_t>(stream)));
}

size_t poetx_forward_workspace_size(int d_in, int d_out, int b, int64_t tokens,
                                    poetx_dtype dtype) {
  const bool is_bf16 = dtype == POETX_BF16;
  if (check_dims(d_in, b, is_bf16) != POETX_OK || check_dims(d_out, b, is_bf16) != POETX_OK ||
      check_common(b, 0, tokens, dtype) != POETX_OK)
    return 0;
  Carver c(nullptr);
  carve_forward(c, d_in, d_out, b, tokens, is_bf16, true);
  return c.off;
}

poetx_status poetx_forward(const void* x, const void* W0, const void* P_blocks,
                           const void* R_blocks, void* y, void* v_saved, int d_in, int d_out,
                           int b, int64_t tokens, poetx_dtype dtype, void* workspace,
                           size_t workspace_bytes, poetx_stream stream) {
  const bool is_bf16 = dtype == POETX_BF16;
  poetx_status st = check_common(b, 0, tokens, dtype);
  if (st != POETX_OK) return st;
  if ((st = check_dims(d_in, b, is_bf16)) != POETX_OK) return st;
  if ((st = check_dims(d_out, b, is_bf16)) != POETX_OK) return st;
  if (tokens == 0) return POETX_OK;  // nothing to compute; pointers may be empty
  if (x == nullptr || W0 == nullptr || P_blocks == nullptr || R_blocks == nullptr ||
      y == nullptr)
    return POETX_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(W0) || !aligned16(P_blocks) || !aligned16(R_blocks) ||
      !aligned16(y) || !aligned16(v_saved))
    return POETX_ERR_INVALID_ARG;
  Carver c(workspace);
  FwdPlan p = carve_forward(c, d_in, d_out, b, tokens, is_bf16, v_saved == nullptr);
  if (workspace == nullptr || c.off > workspace_bytes || !aligned16(workspace))
    return POETX_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  const void* psb = superblocks_or_blocks(P_blocks, p.sb.psb, d_in, b, is_bf16, s, &e);
  if (e != cudaSuccess) return POETX_ERR_CUDA;
  const void* rsb = superblocks_or_blocks(R_blocks, p.sb.rsb, d_out, b, is_bf16, s, &e);
  if (e != cudaSuccess) return POETX_ERR_CUDA;
  if (fuse_block_epilogue(is_bf16, b)) {  // u = P x; v = W0 u and y = R v in one GEMM
    e = tc_transform(static_cast<const bf16*>(x), static_cast<const bf16*>(psb),
                     static_cast<bf16*>(p.sb.u), d_in, 256, tokens, false, "transform", s);
    if (e != cudaSuccess) return POETX_ERR_CUDA;
    return to_status(tc_w0_block(static_cast<const bf16*>(p.sb.u), static_cast<const bf16*>(W0),
                                 static_cast<const bf16*>(rsb), static_cast<bf16*>(v_saved),
                                 static_cast<bf16*>(y), d_in, d_out, tokens, false, s));
  }
  if (!is_bf16 && simt_fused_fits(b))  // u = P x on the fly, v = W0 u, y = R v: one launch
    return to_status(simt_fused_run(static_cast<const float*>(x), static_cast<const float*>(psb),
                                    false, static_cast<const float*>(W0), 1, d_in,
                                    static_cast<const float*>(rsb), false,
                                    static_cast<float*>(v_saved), static_cast<float*>(y),
                                    static_cast<int>(tokens), d_out, d_in, b, "gemm_w0_fused",
                                    s));
  void* v = v_saved != nullptr ? v_saved : p.sb.v;
  e = run_forward_uv(x, W0, psb, p.sb.u, v, d_in, d_out, b, tokens, is_bf16, s);
  if (e != cudaSuccess) return POETX_ERR_CUDA;
  if (is_bf16)
    e = tc_transform(static_cast<const bf16*>(v), static_cast<const bf16*>(rsb),
                     static_cast<bf16*>(y), d_out, superblock(b), tokens, false, "transform", s);
  else
    e = simt_transform(static_cast<const float*>(v), static_cast<const float*>(rsb),
                       static_cast<float*>(y), d_out, b, tokens, false, "transform", s);
  return to_status(e);
}

size_t poetx_backward_workspace_size(int d_in, int d_out, int b, int k, int64_t tokens,
                                     poetx_dtype dtype, int recompute_v) {
  const bool is_bf16 = dtype == POETX_BF16;
  if (check_dims(d_in, b, is_bf16) != POETX_OK || check_dims(d_out, b, is_bf16) != POETX_OK ||
      check_common(b, k, tokens, dtype) != POETX_OK)
    return 0;
  Carver c(nullptr);
  // enough for either form of the backward (block factor fused or not)
  Carver c2(nullptr);
  carve_backward(c, d_in, d_out, b, k, tokens, is_bf16, recompute_v != 0, false);
  carve_backward(c2, d_in, d_out, b, k, tokens, is_bf16, recompute_v != 0, true);
  return c.off > c2.off ? c.off : c2.off;
}

poetx_status poetx_backward(const void* dy, const void* x, const void* W0, const float* theta_P,
                            const float* theta_R, const void* P_blocks, const void* R_blocks,
                            const void* v_saved, void* dx, float* dtheta_P, float* dtheta_R,
                            int d_in, int d_out, int b, int k, int64_t tokens, poetx_dtype dtype,
                            void* workspace, size_t workspace_bytes, poetx_stream stream) {
  const bool is_bf16 = dtype == POETX_BF16;
  poetx_status st = check_common(b, k, tokens, dtype);
  if (st != POETX_OK) return st;
  if ((st = check_dims(d_in, b, is_bf16)) != POETX_OK) return st;
  if ((st = check_dims(d_out, b, is_bf16)) != POETX_OK) return st;
  if (dtheta_P == nullptr || dtheta_R == nullptr || !aligned16(dtheta_P) || !aligned16(dtheta_R))
    return POETX_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (tokens == 0) {  // empty sums: zero gradients; activation pointers may be empty
    if (cudaMemsetAsync(dtheta_P, 0, poetx_packed_size(d_in, b) * sizeof(float), s) !=
            cudaSuccess ||
        cudaMemsetAsync(dtheta_R, 0, poetx_packed_size(d_out, b) * sizeof(float), s) !=
            cudaSuccess)
      return POETX_ERR_CUDA;
    return POETX_OK;
  }
  const void* ptrs[] = {dy, x, W0, theta_P, theta_R, P_blocks, R_blocks, dx};
  for (const void* q : ptrs)
    if (q == nullptr || !aligned16(q)) return POETX_ERR_INVALID_ARG;
  if (!aligned16(v_saved)) return POETX_ERR_INVALID_ARG;
  const bool recompute = v_saved == nullptr;
  const bool fused = fuse_block_epilogue(is_bf16, b);
  Carver c(workspace);
  BwdPlan p = carve_backward(c, d_in, d_out, b, k, tokens, is_bf16, recompute, fused);
  if (workspace == nullptr || c.off > workspace_bytes || !aligned16(workspace))
    return POETX_ERR_WORKSPACE;
  cudaError_t e;
  const void* psb = superblocks_or_blocks(P_blocks, p.sb.psb, d_in, b, is_bf16, s, &e);
  if (e != cudaSuccess) return POETX_ERR_CUDA;
  const void* rsb = superblocks_or_blocks(R_blocks, p.sb.rsb, d_out, b, is_bf16, s, &e);
  if (e != cudaSuccess) return POETX_ERR_CUDA;
  const void* v = v_saved;
  const bool fused32 = !is_bf16 && simt_fused_fits(b);  // fp32: the factors fused into W0's GEMMs
  if (recompute) {
    if (fused32)  // v = W0 (P x), u formed on the fly
      e = simt_fused_run(static_cast<const float*>(x), static_cast<const float*>(psb), false,
                         static_cast<const float*>(W0), 1, d_in, nullptr, false,
                         static_cast<float*>(p.sb.v), nullptr, static_cast<int>(tokens), d_out,
                         d_in, b, "gemm_w0_fused", s);
    else
      e = run_forward_uv(x, W0, psb, p.sb.u, p.sb.v, d_in, d_out, b, tokens, is_bf16, s);
    if (e != cudaSuccess) return POETX_ERR_CUDA;
    v = p.sb.v;
  }
  const int S = superblock(b);
  const bool chain = use_chain(is_bf16, (d_in + d_out) / b, b, k);
  const long long off_R = static_cast<long long>(d_in) * b;  // R blocks follow the P blocks
  if (use_transform_sum(is_bf16, (d_in + d_out) / b, b, k)) {
    // dv = dy R with the G_R^T partials (sum_t v_t dy_t^T) in one pass over dy
    e = tc_transform_sum(static_cast<const bf16*>(dy), static_cast<const bf16*>(v),
                         static_cast<const bf16*>(rsb), static_cast<bf16*>(p.sb.dv), p.part_out,
                         d_out, tokens, p.splits_out, s);
    if (e != cudaSuccess) return POETX_ERR_CUDA;
    if (fused) {
      // du = dv W0 and dx = du P in one GEMM; then the G_P^T partials
      // (sum_t x_t du_t^T) from du and x
      e = tc_w0_block(static_cast<const bf16*>(p.sb.dv), static_cast<const bf16*>(W0),
                      static_cast<const bf16*>(psb), static_cast<bf16*>(p.sb.du),
                      static_cast<bf16*>(dx), d_in, d_out, tokens, true, s);
      if (e != cudaSuccess) return POETX_ERR_CUDA;
      e = tc_outer(static_cast<const bf16*>(x), static_cast<const bf16*>(p.sb.du), p.sb.part,
                   d_in, S, tokens, p.splits_in, s);
      if (e != cudaSuccess) return POETX_ERR_CUDA;
    } else {
      e = tc_w0(static_cast<const bf16*>(p.sb.dv), static_cast<const bf16*>(W0),
                static_cast<bf16*>(p.sb.du), d_in, d_out, tokens, true, s);
      if (e != cudaSuccess) return POETX_ERR_CUDA;
      // dx = du P with the G_P^T partials (sum_t x_t du_t^T) in one pass over du
      e = tc_transform_sum(static_cast<const bf16*>(p.sb.du), static_cast<const bf16*>(x),
                           static_cast<const bf16*>(psb), static_cast<bf16*>(dx), p.sb.part,
                           d_in, tokens, p.splits_in, s);
      if (e != cudaSuccess) return POETX_ERR_CUDA;
    }
    return to_status(chain_adjoint_from_parts(theta_P, d_in / b, p.sb.part, p.splits_in,
                                              theta_R, d_out / b, p.part_out, p.splits_out, b, k,
                                              p.cnp, dtheta_P, dtheta_R, s));
  }
  if (fused32) {
    // dv = dy R on the fly, du = dv W0 (kept for G_P) and dx = du P in one
    // launch; then G_P = sum_t du_t x_t^T and G_R = sum_t dy_t v_t^T
    e = simt_fused_run(static_cast<const float*>(dy), static_cast<const float*>(rsb), true,
                       static_cast<const float*>(W0), d_in, 1, static_cast<const float*>(psb), true,
                       static_cast<float*>(p.sb.du), static_cast<float*>(dx),
                       static_cast<int>(tokens), d_in, d_out, b, "gemm_w0_dgrad_fused", s);
    if (e != cudaSuccess) return POETX_ERR_CUDA;
    // G_P (P blocks first) and G_R in one launch
    e = launch_small_outer2(static_cast<const float*>(p.sb.du), static_cast<const float*>(x),
                            p.cnp.g32[0], d_in, static_cast<const float*>(dy),
                            static_cast<const float*>(v), p.cnp.g32[0] + off_R, d_out, b, tokens,
                            s);
    if (e != cudaSuccess) return POETX_ERR_CUDA;
    return to_status(run_cnp_backward(theta_P, d_in / b, theta_R, d_out / b, b, k, is_bf16,
                                      p.cnp, dtheta_P, dtheta_R, s));
  }
  // R side: dv = dy R, G_R = sum_t dy_t v_t^T
  if (is_bf16)
    e = tc_transform(static_cast<const bf16*>(dy), static_cast<const bf16*>(rsb),
                     static_cast<bf16*>(p.sb.dv), d_out, S, tokens, true, "transform_t", s);
  else
    e = simt_transform(static_cast<const float*>(dy), static_cast<const float*>(rsb),
                       static_cast<float*>(p.sb.dv), d_out, b, tokens, true, "transform_t", s);
  if (e != cudaSuccess) return POETX_ERR_CUDA;
  if (chain)  // G_R^T partials: sum_t v_t dy_t^T per block
    e = tc_outer(static_cast<const bf16*>(v), static_cast<const bf16*>(dy), p.part_out, d_out,
                 S, tokens, p.splits_out, s);
  else
    e = block_gradient(dy, v, d_out, b, tokens, is_bf16, p.sb.part, p.splits_out,
                       p.cnp.g32[0] + off_R, p.cnp.g16[0] ? p.cnp.g16[0] + off_R : nullptr, s);
  if (e != cudaSuccess) return POETX_ERR_CUDA;
  // du = dv W0, and dx = du P (in the same GEMM's epilogue when it fuses)
  if (fused)
    e = tc_w0_block(static_cast<const bf16*>(p.sb.dv), static_cast<const bf16*>(W0),
                    static_cast<const bf16*>(psb), static_cast<bf16*>(p.sb.du),
                    static_cast<bf16*>(dx), d_in, d_out, tokens, true, s);
  else if (is_bf16)
    e = tc_w0(static_cast<const bf16*>(p.sb.dv), static_cast<const bf16*>(W0),
              static_cast<bf16*>(p.sb.du), d_in, d_out, tokens, true, s);
  else
    e = simt_w0(static_cast<const float*>(p.sb.dv), static_cast<const float*>(W0),
                static_cast<float*>(p.sb.du), d_in, d_out, tokens, true, s);
  if (e != cudaSuccess) return POETX_ERR_CUDA;
  // P side: dx = du P, G_P = sum_t du_t x_t^T
  if (fused)
    e = cudaSuccess;
  else if (is_bf16)
    e = tc_transform(static_cast<const bf16*>(p.sb.du), static_cast<const bf16*>(psb),
                     static_cast<bf16*>(dx), d_in, S, tokens, true, "transform_t", s);
  else
    e = simt_transform(static_cast<const float*>(p.sb.du), static_cast<const float*>(psb),
                       static_cast<float*>(dx), d_in, b, tokens, true, "transform_t", s);
  if (e != cudaSuccess) return POETX_ERR_CUDA;
  if (chain) {  // G_P^T partials, then the whole adjoint of both sides in one launch
    e = tc_outer(static_cast<const bf16*>(x), static_cast<const bf16*>(p.sb.du), p.sb.part, d_in,
                 S, tokens, p.splits_in, s);
    if (e != cudaSuccess) return POETX_ERR_CUDA;
    return to_status(chain_adjoint_from_parts(theta_P, d_in / b, p.sb.part, p.splits_in,
                                              theta_R, d_out / b, p.part_out, p.splits_out, b, k,
                                              p.cnp, dtheta_P, dtheta_R, s));
  }
  e = block_gradient(p.sb.du, x, d_in, b, tokens, is_bf16, p.sb.part, p.splits_in,
                     p.cnp.g32[0], p.cnp.g16[0], s);
  if (e != cudaSuccess) return POETX_ERR_CUDA;
  // adjoint of the block build for both sides at once
  return to_status(run_cnp_backward(theta_P, d_in / b, theta_R, d_out / b, b, k, is_bf16, p.cnp,
                                    dtheta_P, dtheta_R, s));
}

size_t poetx_transform_workspace_size(int d, int b, int k, int64_t tokens, poetx_dtype dtype) {
  const bool is_bf16 = dtype == POETX_BF16;
  if (check_dims(d, b, is_bf16) != POETX_OK || check_common(b, k, tokens, dtype) != POETX_OK)
    return 0;
  Carver c(nullptr);
  if (is_bf16 && b < 256) c.take<bf16>(static_cast<size_t>(d) * 256);
  if (is_bf16) {
    const int S = superblock(b);
    const int splits = use_transform_sum(is_bf16, d / b, b, k) ? transform_sum_splits(d, tokens)
                                                               : outer_splits(d, S, tokens);
    c.take<float>(static_cast<size_t>(splits) * d * S);
  }
  carve_cnp(c, d / b, b, k, is_bf16);
  return c.off;
}

poetx_status poetx_transform_forward(const void* x, const void* blocks, void* out, int d, int b,
                                     int64_t tokens, poetx_dtype dtype, void* workspace,
                                     size_t workspace_bytes, poetx_stream stream) {
  const bool is_bf16 = dtype == POETX_BF16;
  poetx_status st = check_common(b, 0, tokens, dtype);
  if (st != POETX_OK) return st;
  if ((st = check_dims(d, b, is_bf16)) != POETX_OK) return st;
  if (tokens == 0) return POETX_OK;
  if (x == nullptr || blocks == nullptr || out == nullptr || !aligned16(x) ||
      !aligned16(blocks) || !aligned16(out))
    return POETX_ERR_INVALID_ARG;
  Carver c(workspace);
  bf16* sbuf = (is_bf16 && b < 256) ? c.take<bf16>(static_cast<size_t>(d) * 256) : nullptr;
  if (c.off > 0 && (workspace == nullptr || c.off > workspace_bytes || !aligned16(workspace)))
    return POETX_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  const void* sb = superblocks_or_blocks(blocks, sbuf, d, b, is_bf16, s, &e);
  if (e != cudaSuccess) return POETX_ERR_CUDA;
  if (is_bf16)
    e = tc_transform(static_cast<const bf16*>(x), static_cast<const bf16*>(sb),
                     static_cast<bf16*>(out), d, superblock(b), tokens, false, "transform", s);
  else
    e = simt_transform(static_cast<const float*>(x), static_cast<const float*>(sb),
                       static_cast<float*>(out), d, b, tokens, false, "transform", s);
  return to_status(e);
}

poetx_status poetx_transform_backward(const void* dout, const void* x, const float* theta,
                                      const void* blocks, void* dx, float* dtheta, int d, int b,
                                      int k, int64_t tokens, poetx_dtype dtype, void* workspace,
                                      size_t workspace_bytes, poetx_stream stream) {
  const bool is_bf16 = dtype == POETX_BF16;
  poetx_status st = check_common(b, k, tokens, dtype);
  if (st != POETX_OK) return st;
  if ((st = check_dims(d, b, is_bf16)) != POETX_OK) return st;
  if (dtheta == nullptr || !aligned16(dtheta)) return POETX_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (tokens == 0)
    return to_status(cudaMemsetAsync(dtheta, 0, poetx_packed_size(d, b) * sizeof(float), s));
  const void* ptrs[] = {dout, x, theta, blocks, dx};
  for (const void* q : ptrs)
    if (q == nullptr || !aligned16(q)) return POETX_ERR_INVALID_ARG;
  Carver c(workspace);
  bf16* sbuf = (is_bf16 && b < 256) ? c.take<bf16>(static_cast<size_t>(d) * 256) : nullptr;
  const int S = superblock(b);
  const bool ts = use_transform_sum(is_bf16, d / b, b, k);
  const int splits =
      !is_bf16 ? 1 : (ts ? transform_sum_splits(d, tokens) : outer_splits(d, S, tokens));
  float* part = is_bf16 ? c.take<float>(static_cast<size_t>(splits) * d * S) : nullptr;
  CnpBufs cnp = carve_cnp(c, d / b, b, k, is_bf16);
  if (workspace == nullptr || c.off > workspace_bytes || !aligned16(workspace))
    return POETX_ERR_WORKSPACE;
  cudaError_t e;
  const void* sb = superblocks_or_blocks(blocks, sbuf, d, b, is_bf16, s, &e);
  if (e != cudaSuccess) return POETX_ERR_CUDA;
  if (ts) {  // dx = dout B with the G^T partials (sum_t x_t dout_t^T) in one pass
    e = tc_transform_sum(static_cast<const bf16*>(dout), static_cast<const bf16*>(x),
                         static_cast<const bf16*>(sb), static_cast<bf16*>(dx), part, d, tokens,
                         splits, s);
    if (e != cudaSuccess) return POETX_ERR_CUDA;
    return to_status(chain_adjoint_from_parts(theta, d / b, part, splits, nullptr, 0, nullptr, 1,
                                              b, k, cnp, dtheta, nullptr, s));
  }
  if (is_bf16)
    e = tc_transform(static_cast<const bf16*>(dout), static_cast<const bf16*>(sb),
                     static_cast<bf16*>(dx), d, S, tokens, true, "transform_t", s);
  else
    e = simt_transform(static_cast<const float*>(dout), static_cast<const float*>(sb),
                       static_cast<float*>(dx), d, b, tokens, true, "transform_t", s);
  if (e != cudaSuccess) return POETX_ERR_CUDA;
  if (use_chain(is_bf16, d / b, b, k)) {  // G^T partials, then the adjoint in one launch
    e = tc_outer(static_cast<const bf16*>(x), static_cast<const bf16*>(dout), part, d, S, tokens,
                 splits, s);
    if (e != cudaSuccess) return POETX_ERR_CUDA;
    return to_status(chain_adjoint_from_parts(theta, d / b, part, splits, nullptr, 0, nullptr, 1,
                                              b, k, cnp, dtheta, nullptr, s));
  }
  e = block_gradient(dout, x, d, b, tokens, is_bf16, part, splits, cnp.g32[0], cnp.g16[0], s);
  if (e != cudaSuccess) return POETX_ERR_CUDA;
  return to_status(
      run_cnp_backward(theta, d / b, nullptr, 0, b, k, is_bf16, cnp, dtheta, nullptr, s));
}

poetx_status poetx_device_status(void) {
  if (cudaDeviceSynchronize() != cudaSuccess) return POETX_ERR_CUDA;
  const int v = read_and_clear_device_status();
  if (v < 0) return POETX_ERR_CUDA;
  return v == 0 ? POETX_OK : static_cast<poetx_status>(v);
}

long long poetx_launch_count(void) { return g_launches.load(); }

int poetx_profile_start(int capacity) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  g_prof_recs.clear();
  g_prof_used = 0;
  while (static_cast<int>(g_prof_pool.size()) < 2 * capacity) {
    cudaEvent_t ev;
    if (cudaEventCreate(&ev) != cudaSuccess) return -1;
    g_prof_pool.push_back(ev);
  }
  g_prof_on = true;
  return 0;
}

void poetx_profile_stop(void) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  g_prof_on = false;
}

int poetx_profile_query(const char* tag, int* count, double* total_ms) {
  std::lock_guard<std::mutex> lock(g_prof_mu);
  int n = 0;
  double total = 0.0;
  for (const ProfRecord& r : g_prof_recs) {
    if (!r.closed) continue;
    if (tag != nullptr && std::strcmp(tag, r.tag) != 0) continue;
    if (cudaEventSynchronize(r.stop) != cudaSuccess) return -1;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess) return -1;
    total += ms;
    ++n;
  }
  if (count != nullptr) *count = n;
  if (total_ms != nullptr) *total_ms = total;
  return 0;
}

poetx_status poetx_build_blocks_noalloc(const float* theta, int d, int b, int k, poetx_dtype dtype,
                                        void* blocks, poetx_stream stream) {
  const bool is_bf16 = dtype == POETX_BF16;
  poetx_status st = check_common(b, k, 0, dtype);
  if (st != POETX_OK) return st;
  if ((st = check_dims(d, b, is_bf16)) != POETX_OK) return st;
  if (theta == nullptr || blocks == nullptr || !aligned16(theta) || !aligned16(blocks))
    return POETX_ERR_INVALID_ARG;
  if (static_cast<long long>(d) * b > kNoAllocMaxElems) return POETX_ERR_WORKSPACE;
  Carver dry(nullptr);
  carve_build(dry, d / b, b, k, is_bf16);
  if (dry.off > kNoAllocScratchBytes) return POETX_ERR_WORKSPACE;
  void* scratch = build_scratch_address(static_cast<cudaStream_t>(stream));
  if (scratch == nullptr) return POETX_ERR_CUDA;
  Carver c(scratch);
  BuildBufs w = carve_build(c, d / b, b, k, is_bf16);
  return to_status(
      run_build(theta, d / b, b, k, is_bf16, blocks, w, static_cast<cudaStream_t>(stream)));
}

// The index-map kernel keeps one 8-byte entry per feature (4 bf16 or 2 fp32
// rows interleaved) in at most 224 KiB of shared memory.
constexpr int kMaxPermuteFeatures = 28672;

poetx_status poetx_permute_features(const void* in, const int32_t* perm, void* out, int64_t rows,
                                    int d, poetx_dtype dtype, poetx_stream stream) {
  const bool is_bf16 = dtype == POETX_BF16;
  if (dtype != POETX_F32 && dtype != POETX_BF16) return POETX_ERR_INVALID_ARG;
  if (rows < 0 || d <= 0 || (d * (is_bf16 ? 2 : 4)) % 16 != 0 || d > kMaxPermuteFeatures)
    return POETX_ERR_INVALID_ARG;
  if (rows == 0) return POETX_OK;
  if (in == nullptr || perm == nullptr || out == nullptr || in == out || !aligned16(in) ||
      !aligned16(out) || !aligned16(perm))  // the column map is read as 16-byte vectors
    return POETX_ERR_INVALID_ARG;
  return to_status(launch_permute_rows(in, rows, nullptr, perm, out, rows, d, is_bf16,
                                       static_cast<cudaStream_t>(stream)));
}

poetx_status poetx_fold_permutations(const void* W0, const int32_t* perm_out,
                                     const int32_t* perm_in, void* W0_folded, int d_in,
                                     int d_out, poetx_dtype dtype, poetx_stream stream) {
  const bool is_bf16 = dtype == POETX_BF16;
  if (dtype != POETX_F32 && dtype != POETX_BF16) return POETX_ERR_INVALID_ARG;
  if (d_in <= 0 || d_out <= 0 || (d_in * (is_bf16 ? 2 : 4)) % 16 != 0 ||
      d_in > kMaxPermuteFeatures)
    return POETX_ERR_INVALID_ARG;
  if (W0 == nullptr || perm_out == nullptr || perm_in == nullptr || W0_folded == nullptr ||
      W0 == W0_folded || !aligned16(W0) || !aligned16(W0_folded) ||
      (reinterpret_cast<uintptr_t>(perm_out) & 3u) != 0 || !aligned16(perm_in))
    return POETX_ERR_INVALID_ARG;
  return to_status(launch_permute_rows(W0, d_out, perm_out, perm_in, W0_folded, d_out, d_in,
                                       is_bf16, static_cast<cudaStream_t>(stream)));
}

size_t poetx_merge_workspace_size(int d_in, int d_out, int b, poetx_dtype dtype) {
  const bool is_bf16 = dtype == POETX_BF16;
  if (check_dims(d_in, b, is_bf16) != POETX_OK || check_dims(d_out, b, is_bf16) != POETX_OK ||
      check_common(b, 0, 0, dtype) != POETX_OK)
    return 0;
  Carver c(nullptr);
  c.take<char>(static_cast<size_t>(d_out) * d_in * elem_size(is_bf16));
  if (is_bf16 && b < 256) {
    c.take<bf16>(static_cast<size_t>(d_in) * 256);
    c.take<bf16>(static_cast<size_t>(d_out) * 256);
  }
  return c.off;
}

poetx_status poetx_merge(const void* W0, const void* P_blocks, const void* R_blocks, void* W0_out,
                         float* theta_P, float* theta_R, int d_in, int d_out, int b,
                         poetx_dtype dtype, void* workspace, size_t workspace_bytes,
                         poetx_stream stream) {
  const bool is_bf16 = dtype == POETX_BF16;
  poetx_status st = check_common(b, 0, 0, dtype);
  if (st != POETX_OK) return st;
  if ((st = check_dims(d_in, b, is_bf16)) != POETX_OK) return st;
  if ((st = check_dims(d_out, b, is_bf16)) != POETX_OK) return st;
  const void* ptrs[] = {W0, P_blocks, R_blocks, W0_out};
  for (const void* q : ptrs)
    if (q == nullptr || !aligned16(q)) return POETX_ERR_INVALID_ARG;
  if (!aligned16(theta_P) || !aligned16(theta_R)) return POETX_ERR_INVALID_ARG;
  Carver c(workspace);
  void* M = c.take<char>(static_cast<size_t>(d_out) * d_in * elem_size(is_bf16));
  bf16* psb = nullptr;
  bf16* rsb = nullptr;
  if (is_bf16 && b < 256) {
    psb = c.take<bf16>(static_cast<size_t>(d_in) * 256);
    rsb = c.take<bf16>(static_cast<size_t>(d_out) * 256);
  }
  if (workspace == nullptr || c.off > workspace_bytes || !aligned16(workspace))
    return POETX_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  const void* P = superblocks_or_blocks(P_blocks, psb, d_in, b, is_bf16, s, &e);
  if (e != cudaSuccess) return POETX_ERR_CUDA;
  const void* R = superblocks_or_blocks(R_blocks, rsb, d_out, b, is_bf16, s, &e);
  if (e != cudaSuccess) return POETX_ERR_CUDA;
  if (is_bf16) {
    const int S = superblock(b);
    // M = W0 P: W0's rows through the transposed block transform
    e = tc_transform(static_cast<const bf16*>(W0), static_cast<const bf16*>(P),
                     static_cast<bf16*>(M), d_in, S, d_out, true, "merge", s);
    if (e != cudaSuccess) return POETX_ERR_CUDA;
    // W0_out = R M: one S x S block of R times S rows of M per batch
    TcGemm g;
    g.M = S;
    g.N = d_in;
    g.K = S;
    g.batches = d_out / S;
    g.BN = 256;
    g.A = op(R, d_out, S, S, false, S, 0);     // A[m][kk] = R_g[m][kk]
    g.B = op(M, d_out, d_in, d_in, true, 0, S);  // B[n][kk] = M[g*S + kk][n]
    g.epi.out_bf16 = static_cast<bf16*>(W0_out);
    g.epi.ld = d_in;
    g.epi.row_g = S;
    g.epi.out_rows = d_out;
    g.tag = "merge";
    e = tc_gemm_run(g, s);
  } else {
    e = simt_transform(static_cast<const float*>(W0), static_cast<const float*>(P),
                       static_cast<float*>(M), d_in, b, d_out, true, "merge", s);
    if (e != cudaSuccess) return POETX_ERR_CUDA;
    SimtGemm g;
    g.M = b;
    g.N = d_in;
    g.K = b;
    g.batches = d_out / b;
    g.A = R;
    g.a_g = static_cast<long long>(b) * b;
    g.a_m = b;
    g.a_k = 1;
    g.B = M;
    g.b_g = static_cast<long long>(b) * d_in;
    g.b_k = d_in;
    g.b_n = 1;
    g.epi.out_f32 = static_cast<float*>(W0_out);
    g.epi.ld = d_in;
    g.epi.row_g = b;
    g.tag = "merge";
    e = simt_gemm_run(g, s);
  }
  if (e != cudaSuccess) return POETX_ERR_CUDA;
  if (theta_P != nullptr &&
      cudaMemsetAsync(theta_P, 0, poetx_packed_size(d_in, b) * sizeof(float), s) != cudaSuccess)
    return POETX_ERR_CUDA;
  if (theta_R != nullptr &&
      cudaMemsetAsync(theta_R, 0, poetx_packed_size(d_out, b) * sizeof(float), s) != cudaSuccess)
    return POETX_ERR_CUDA;
  return POETX_OK;
}

poetx_status poetx_adam_update(float* theta, const float* grad, float* m, float* v, int64_t n,
                               int step, float lr, float beta1, float beta2, float eps,
                               float weight_decay, poetx_stream stream) {
  if (n < 0 || step < 1 || !(beta1 >= 0.f && beta1 < 1.f) || !(beta2 >= 0.f && beta2 < 1.f) ||
      !(eps > 0.f))
    return POETX_ERR_INVALID_ARG;
  if (n == 0) return POETX_OK;
  if (theta == nullptr || grad == nullptr || m == nullptr || v == nullptr)
    return POETX_ERR_INVALID_ARG;
  const double bc1 = 1.0 - std::pow(static_cast<double>(beta1), step);
  const double bc2 = 1.0 - std::pow(static_cast<double>(beta2), step);
  return to_status(launch_adam(theta, grad, m, v, n, lr, beta1, beta2, eps, weight_decay,
                               static_cast<float>(bc1), static_cast<float>(bc2),
                               static_cast<cudaStream_t>(stream)));
}

poetx_status poetx_quantize_w0(const void* W0, int8_t* W0_q, float* scales, int d_in, int d_out,
                               poetx_dtype dtype, poetx_stream stream) {
  if (dtype != POETX_F32 && dtype != POETX_BF16) return POETX_ERR_INVALID_ARG;
  if (d_in < 0 || d_out < 0) return POETX_ERR_INVALID_ARG;
  if (d_in == 0 || d_out == 0) return POETX_OK;
  if (W0 == nullptr || W0_q == nullptr || scales == nullptr) return POETX_ERR_INVALID_ARG;
  return to_status(launch_quantize_rows(W0, dtype == POETX_BF16, W0_q, scales, d_in, d_out,
                                        static_cast<cudaStream_t>(stream)));
}

poetx_status poetx_dequantize_w0(const int8_t* W0_q, const float* scales, void* W0, int d_in,
                                 int d_out, poetx_dtype dtype, poetx_stream stream) {
  if (dtype != POETX_F32 && dtype != POETX_BF16) return POETX_ERR_INVALID_ARG;
  if (d_in < 0 || d_out < 0) return POETX_ERR_INVALID_ARG;
  if (d_in == 0 || d_out == 0) return POETX_OK;
  if (W0 == nullptr || W0_q == nullptr || scales == nullptr) return POETX_ERR_INVALID_ARG;
  return to_status(launch_dequantize(W0_q, scales, W0, dtype == POETX_BF16, d_in, d_out,
                                     static_cast<cudaStream_t>(stream)));
}

int poetx_set_block_epilogue_fusion(int enable) {
  return g_fuse_block_epilogue.exchange(enable != 0 ? 1 : 0);
}

int poetx_set_w0_split_tail(int enable) {
  return g_w0_split_tail.exchange(enable != 0 ? 1 : 0);
}

int poetx_set_w0_pair_mma(int enable) { return g_w0_pair.exchange(enable != 0 ? 1 : 0); }

}  // extern "C"





