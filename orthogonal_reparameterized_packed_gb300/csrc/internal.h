// Internal interfaces shared by the library's translation units.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace poetx {

// Launch with programmatic stream serialization: the kernel may start
// before its predecessor on `s` has finished; every kernel of the library
// calls pdl_wait() before it touches global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Where a contraction's result goes: for batch g, K-split s, row r and
// column c of the (batch-local) result,
//   v   = alpha * acc + beta * X[off] + gamma * Y[off] + delta * (r == c)
//   off = (g * row_g + s * row_s + r) * ld + g * col_g + c
// and v is stored to out_f32[off] and/or out_bf16[off].  Rows r >=
// row_limit are skipped.  X, Y, out_f32, out_bf16 may each be null.
// out_rows x ld is the extent of the output array (used for TMA stores).
struct EpiArgs {
  float alpha = 1.f;
  const float* X = nullptr;
  float beta = 0.f;
  const float* Y = nullptr;
  float gamma = 0.f;
  float delta = 0.f;
  float* out_f32 = nullptr;
  __nv_bfloat16* out_bf16 = nullptr;
  long long ld = 0;
  int row_g = 0, row_s = 0, col_g = 0;
  int row_limit = 0x7fffffff;
  long long out_rows = 0;
};

// ---------------------------------------------------------------- tcgen05
// C = A * B^T per batch on the tensor cores (bf16 in, fp32 accumulate).
// Each operand is a window of a 2-D row-major bf16 array:
//   major K : array rows index M (or N), columns index K
//   major MN: array rows index K, columns index M (or N)
// For batch g the window starts at M/N coordinate g*mn_per_g and K
// coordinate g*k_per_g.  Reads past the array's extent return zeros.
struct TcOperand {
  const void* ptr = nullptr;
  long long rows = 0, cols = 0, pitch = 0;  // pitch in elements
  bool mn_major = false;
  int mn_per_g = 0, k_per_g = 0;
};

struct TcGemm {
  int M = 0, N = 0, K = 0;  // per batch
  int batches = 1;
  int splits = 1;           // K is split; split s writes rows s * epi.row_s on
  int BN = 256;             // 128 or 256
  // Keep the B operand of a (batch, N tile) resident in shared memory while
  // the CTA walks consecutive M tiles (needs splits == 1 and BN*K*2 <= 128 KiB).
  bool b_resident = false;
  // W0 GEMMs: run as clusters of two CTAs on adjacent M tiles (needed by
  // split_tail, whose partial sums move between the two CTAs)
  bool cluster2 = false;
  // cluster2: when the last round of tiles would leave clusters idle, spread
  // its tiles one per cluster, the two CTAs summing halves of K
  bool split_tail = false;
  TcOperand A, B;
  EpiArgs epi;
  // Block-diagonal factor in the epilogue (W0 GEMMs, BN = 256): N tile j of
  // the product (written to epi.out_bf16 when that is set) is multiplied by
  // the 256 x 256 block j of `blk` (rows j*256.., same major-ness as B:
  // out_blk[:, j] = C[:, j] * blk_j^T for K-major, C[:, j] * blk_j for
  // MN-major) and written to out_blk with the layout of epi.
  TcOperand blk;
  __nv_bfloat16* out_blk = nullptr;
  const char* tag = "tc_gemm";  // name under which launches are profiled
};

// The transposed block transform and the token sums of the block gradient in
// one pass over X (transform_sum_tc.cu), 256 x 256 superblocks:
//   out[t][g*256+n] = sum_kk X[t][g*256+kk] sb[g*256+kk][n]              (bf16)
//   part[s][g][m][n] = sum_{t in split s} Z[t][g*256+m] X[t][g*256+n]     (fp32)
// `splits` must be transform_sum_splits(d, T).
int transform_sum_splits(int d, long long T);
cudaError_t tc_transform_sum(const __nv_bfloat16* X, const __nv_bfloat16* Z,
                             const __nv_bfloat16* sb, __nv_bfloat16* out, float* part, int d,
                             long long T, int splits, cudaStream_t stream);

// The W0 GEMM (bf16 out, one batch, no K split, A K-major, N a multiple of
// 256) on CTA pairs: 256 x 256 tiles, one tcgen05.mma.cta_group::2 per K
// slice of 16; see gemm_pair.cu.
cudaError_t w0_pair_run(const TcGemm& g, cudaStream_t stream);

// Number of K splits the engine will actually use for `want` splits.
int tc_effective_splits(int K, int want);
cudaError_t tc_gemm_run(const TcGemm& g, cudaStream_t stream);

// ------------------------------------------------------------------- SIMT
// C = A * B per batch on the CUDA cores, fp32 accumulate, arbitrary strides:
//   A(g, m, k) = A[g*a_g + m*a_m + k*a_k], B(g, k, n) = B[g*b_g + k*b_k + n*b_n]
// Inputs are float or bf16 (both operands the same type).
struct SimtGemm {
  int M = 0, N = 0, K = 0, batches = 1;
  int splits = 1;  // set by simt_gemm_run: K slices per output tile (a cluster)
  bool bf16_inputs = false;
  const void* A = nullptr;
  long long a_g = 0, a_m = 0, a_k = 0;
  const void* B = nullptr;
  long long b_g = 0, b_k = 0, b_n = 0;
  EpiArgs epi;
  const char* tag = "simt_gemm";
};
cudaError_t simt_gemm_run(const SimtGemm& g, cudaStream_t stream);
// The fp32 W0 product with block-diagonal factors on both sides in one
// launch (simt_fused_fits(b): b divides 32, or b = 64):
//   C = A W^T-style product with A[t][k] = sum_j X[t][g b + j] L_g(k % b, j),
//   out[t][n] = sum_j C[t][g b + j] R_g(n % b, j); L_g(kl, j) = L_g[kl][j]
//   (or L_g[j][kl] when l_trans), likewise R; B(k, n) = W[k w_k + n w_n].
// C (if not null) is stored; R null: no right factor (out unused).
bool simt_fused_fits(int b);
cudaError_t simt_fused_run(const float* X, const float* L, bool l_trans, const float* W,
                           long long w_k, long long w_n, const float* R, bool r_trans, float* C,
                           float* out, int M, int N, int K, int b, const char* tag,
                           cudaStream_t stream);

// ------------------------------------------------------------ b x b chains
// One cooperative launch per chain of b x b products (tensor cores, b a
// multiple of 128, k <= kChainMaxK); see chain_tc.cu.
constexpr int kChainMaxK = 8;
constexpr int kChainMaxPhases = 20;  // >= 2 * kChainMaxK - 1 product phases

// True when the chain of n blocks of size b and order k runs as one launch
// (b a multiple of 128, k <= kChainMaxK, at most two persistent D tiles per CTA).
bool chain_fits(int n, int b, int k);

// blocks = (I + Q)(I + Q + ... + Q^k) for the n blocks of one side, bf16 out.
// Scratch [n][b][b] bf16: q_hi, q_lo, e16[0], e16[1]; two_i [b][b] bf16;
// counter [kChainMaxPhases] words.
struct ChainBuildArgs {
  int n = 0, b = 0, k = 0;
  const float* theta = nullptr;
  __nv_bfloat16* q_hi = nullptr;
  __nv_bfloat16* q_lo = nullptr;
  __nv_bfloat16* two_i = nullptr;
  __nv_bfloat16* e16[2] = {nullptr, nullptr};
  unsigned int* counter = nullptr;
  __nv_bfloat16* blocks = nullptr;
};
cudaError_t chain_build(const ChainBuildArgs& a, cudaStream_t stream);

// Packed gradients of both sides from the split-K partials of the TRANSPOSED
// block gradients G^T (blocks [0, n_a) from part_a / theta_a, the rest from
// part_b / theta_b).  Scratch [n_a + n_b][b][b]: q16, e16[2..k], f16[0..1],
// x16 (bf16) and d32 (fp32); two_i [b][b] bf16; counter [kChainMaxPhases] words.
struct ChainAdjointArgs {
  int n_a = 0, n_b = 0, b = 0, k = 0;
  const float* theta_a = nullptr;
  const float* theta_b = nullptr;
  __nv_bfloat16* q16 = nullptr;
  __nv_bfloat16* two_i = nullptr;
  __nv_bfloat16* e16[kChainMaxK + 2] = {};
  __nv_bfloat16* f16[2] = {nullptr, nullptr};
  __nv_bfloat16* x16 = nullptr;  // k = 3: 2Q
  float* d32 = nullptr;
  const float* part_a = nullptr;
  const float* part_b = nullptr;
  int splits_a = 1, splits_b = 1, nsb_a = 0, nsb_b = 0, S = 0;
  float* dtheta_a = nullptr;
  float* dtheta_b = nullptr;
  unsigned int* counter = nullptr;
};
cudaError_t chain_adjoint(const ChainAdjointArgs& a, cudaStream_t stream);

// ------------------------------------------- b x b chains on CTA pairs
// 1 <= k <= 16 and b in {32, 64, 128, 256} (256 x 256 superblocks), bf16
// blocks: one cluster of two CTAs per superblock with every operand in
// shared memory (cnp_pair.cu).  n * b must be a multiple of 256.
bool cnp_pair_fits(int b, int k);
// blocks [n][b][b] = (I + Q)(I + Q + ... + Q^k) from theta [n][b(b-1)/2].
cudaError_t cnp_build_pair(const float* theta, int n, int b, int k, __nv_bfloat16* blocks,
                           cudaStream_t stream);

// Packed gradients of both sides from the split-K partials of the
// TRANSPOSED block gradients G^T over 256 x 256 superblocks (blocks
// [0, n_a) of side a, then n_b of side b).  Scratch: hg
// [(n_a + n_b) * b / 256 * 256][256] bf16.
struct CnpAdjointPairArgs {
  int n_a = 0, n_b = 0, b = 0, k = 3;
  const float* theta_a = nullptr;
  const float* theta_b = nullptr;
  const float* part_a = nullptr;
  const float* part_b = nullptr;
  int splits_a = 1, splits_b = 1;
  __nv_bfloat16* hg = nullptr;
  float* dtheta_a = nullptr;
  float* dtheta_b = nullptr;
};
cudaError_t cnp_adjoint_pair(const CnpAdjointPairArgs& a, cudaStream_t stream);

// ------------------------------------------------------------ elementwise
// Packed parameters of two sides (theta_a: n_a blocks, theta_b: n_b blocks;
// theta_b may be null when n_b = 0) -> Q [n_a + n_b][b][b], fp32 and/or bf16.
cudaError_t launch_unpack(const float* theta_a, int n_a, const float* theta_b, int n_b, int b,
                          float* q_f32, __nv_bfloat16* q_bf16, cudaStream_t s);
// out = Q + I in the requested type (k = 0 blocks).
cudaError_t launch_identity_plus(const float* q, int n, int b, float* out_f32,
                                 __nv_bfloat16* out_bf16, cudaStream_t s);
// blocks [n][b][b] bf16 -> superblocks [n*b/S][S][S] with the b-blocks on
// the diagonal and zeros elsewhere.
cudaError_t launch_expand_superblocks(const __nv_bfloat16* blocks, int n, int b, int S,
                                      __nv_bfloat16* out, cudaStream_t s);
// G[g] = sum_s part[s][sb][off..][off..] (diagonal b-block g of superblock
// sb = g*b/S) -> fp32 and/or bf16 [n][b][b].
cudaError_t launch_reduce_extract(const float* part, int splits, int n, int b, int S,
                                  float* out_f32, __nv_bfloat16* out_bf16, cudaStream_t s);
// dtheta[g][idx(i,j)] = M[g][i][j] - M[g][j][i] with M = A (+ B if B != null),
// for n_a + n_b blocks: the first n_a go to dtheta_a, the rest to dtheta_b.
// Blocks of b <= 64 with every matrix of one block in one CTA's shared
// memory (fp32 arithmetic): the whole build, or the whole adjoint of both
// sides (G = dL/dR per block, [n_a + n_b][b][b] fp32), in one launch.
bool small_chain_fits(int b);
// G[g] = sum_t A[t][g-block]^T B[t][g-block] for fp32 blocks of b <= 64
// (small_chain_fits), [d/b][b][b].
cudaError_t launch_small_outer(const float* A, const float* B, float* G, int d, int b, long long T,
                               cudaStream_t s);
// Both sides in one launch: G0 from (A0, B0) over d0 features, G1 from
// (A1, B1) over d1.
cudaError_t launch_small_outer2(const float* A0, const float* B0, float* G0, int d0,
                                const float* A1, const float* B1, float* G1, int d1, int b,
                                long long T, cudaStream_t s);
cudaError_t launch_small_build(const float* theta, int n, int b, int k, float* out32,
                               __nv_bfloat16* out16, cudaStream_t s);
cudaError_t launch_small_adjoint(const float* theta_a, int n_a, const float* theta_b, int n_b,
                                 int b, int k, const float* G, float* dtheta_a, float* dtheta_b,
                                 cudaStream_t s);
cudaError_t launch_pack_skew(const float* A, const float* B, int n_a, int n_b, int b,
                             float* dtheta_a, float* dtheta_b, cudaStream_t s);
// Tiled elementwise steps of the b x b chains (b a multiple of 32), blocks
// [0, n_a) of side a and [n_a, n_a + n_b) of side b; null outputs are skipped:
//   q_hi (+ q_lo) = bf16 Q (+ bf16 remainder) from theta;  two_i = 2I;
//   f16 (+ f32) = sum over splits of the diagonal b-blocks of the partials.
struct PrepTilesArgs {
  int n_a = 0, n_b = 0, b = 0;
  const float* theta_a = nullptr;
  const float* theta_b = nullptr;
  __nv_bfloat16* q_hi = nullptr;
  __nv_bfloat16* q_lo = nullptr;
  __nv_bfloat16* q_x2 = nullptr;  // if set: 2 * q_hi (exact in bf16)
  __nv_bfloat16* two_i = nullptr;
  const float* part_a = nullptr;
  const float* part_b = nullptr;
  int splits_a = 1, splits_b = 1, nsb_a = 0, nsb_b = 0, S = 0;
  __nv_bfloat16* f16 = nullptr;
  float* f32 = nullptr;
  unsigned int* zero_words = nullptr;  // if set: zeroed (the next chain's barrier counters)
  int n_zero_words = 0;
};
cudaError_t launch_prep_tiles(const PrepTilesArgs& a, cudaStream_t s);
// dtheta = sign * pack(D - D^T) per block.
cudaError_t launch_pack_tiles(const float* D, float sign, int n_a, int n_b, int b,
                              float* dtheta_a, float* dtheta_b, cudaStream_t s);
// out[r][i] = in[row_map ? row_map[r] : r][col_map[i]]; in has in_rows rows
// of d elements, out has rows rows; d * elem_size multiple of 16 and
// d * 8 bytes at most 224 KiB.  Out-of-range map entries give 0 and POETX_ERR_INVALID_ARG in the
// status word.
cudaError_t launch_permute_rows(const void* in, long long in_rows, const int* row_map,
                                const int* col_map, void* out, long long rows, int d,
                                bool is_bf16, cudaStream_t s);
// INT8 frozen weight: per-row codes and scales from W (bf16 or fp32), and back.
cudaError_t launch_quantize_rows(const void* W, bool is_bf16, int8_t* q, float* scales, int d_in,
                                 int d_out, cudaStream_t s);
cudaError_t launch_dequantize(const int8_t* q, const float* scales, void* W, bool is_bf16,
                              int d_in, int d_out, cudaStream_t s);
// theta -= lr * (m_hat / (sqrt(v_hat) + eps) + wd * theta) with updated moments.
cudaError_t launch_adam(float* theta, const float* grad, float* m, float* v, long long n,
                        float lr, float beta1, float beta2, float eps, float wd, float bc1,
                        float bc2, cudaStream_t s);
cudaError_t launch_f32_to_bf16(const float* in, long long count, __nv_bfloat16* out,
                               cudaStream_t s);

// ------------------------------------------------------------ bookkeeping
int* device_status_ptr();            // per-device status word (device memory)
int read_and_clear_device_status();  // synchronous
int sm_count();
// Every kernel launch is bracketed by these: they count launches and, while
// profiling is on, record CUDA events on the launch stream under `tag`.
void prof_begin(const char* tag, cudaStream_t s);
void prof_end(const char* tag, cudaStream_t s);

}  // namespace poetx
