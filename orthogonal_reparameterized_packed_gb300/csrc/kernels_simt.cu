// CUDA-core kernels: the fp32 contraction engine (FFMA; used for every
// contraction in fp32 mode, where tensor-core tf32 would miss the fp32
// tolerance, and for blocks narrower than one 128-wide MMA tile), plus the
// small elementwise kernels of the path (unpack, superblock expansion,
// split-K reduction, skew projection and pack).
#include <mutex>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace poetx {

namespace {

constexpr int TM = 64, TN = 64, TK = 32, SIMT_THREADS = 256;
constexpr int kFusedXW = 64;  // the fused kernel's widest block

template <typename T>
__device__ __forceinline__ float load_f(const T* p, long long i);
template <>
__device__ __forceinline__ float load_f<float>(const float* p, long long i) {
  return p[i];
}
template <>
__device__ __forceinline__ float load_f<__nv_bfloat16>(const __nv_bfloat16* p, long long i) {
  return __bfloat162float(p[i]);
}

// C(g) = A(g) * B(g), 64x64 output tile per CTA, 4x4 per thread, K in steps
// of 32 staged in shared memory; each thread loads its share of the next
// step's operands into registers while the current step's FMAs run.  With
// p.splits > 1 the K range is cut into that many slices, one per CTA of a
// cluster along x (the tile's N index is blockIdx.x / splits); each rank
// finalises a contiguous share of the tile's entries, loading all slices'
// partial values of an entry at once and adding them in rank order (a fixed
// summation order: results do not depend on timing or on which rank adds),
// and applies the epilogue to them.  No global scratch, no atomics.
template <typename T>
__global__ void __launch_bounds__(SIMT_THREADS) simt_gemm_kernel(const SimtGemm p) {
  pdl_wait();
  pdl_trigger();
  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];
  __shared__ float Ps[TM][TN + 1];  // this slice's partial tile (splits > 1)
  const int g = blockIdx.z;
  const int m0 = blockIdx.y * TM;
  const int split = p.splits > 1 ? static_cast<int>(blockIdx.x) % p.splits : 0;
  const int n0 = (p.splits > 1 ? static_cast<int>(blockIdx.x) / p.splits : blockIdx.x) * TN;
  const int kslice = p.splits > 1 ? ((p.K + p.splits * TK - 1) / (p.splits * TK)) * TK : p.K;
  const int k_begin = split * kslice;
  const int k_end = min(p.K, k_begin + kslice);
  const T* A = static_cast<const T*>(p.A) + static_cast<long long>(g) * p.a_g;
  const T* B = static_cast<const T*>(p.B) + static_cast<long long>(g) * p.b_g;
  const int tx = threadIdx.x % 16;  // n direction
  const int ty = threadIdx.x / 16;  // m direction
  float acc[4][4] = {};
  constexpr int PA = TM * TK / SIMT_THREADS, PB = TN * TK / SIMT_THREADS;
  float ra[PA], rb[PB];  // the next K step's operands, loaded during this step's FMAs
  auto fetch = [&](int k0) {
#pragma unroll
    for (int q = 0; q < PA; ++q) {
      const int e = threadIdx.x + q * SIMT_THREADS;
      const int mm = e / TK, kk = e % TK;
      const int m = m0 + mm, k = k0 + kk;
      ra[q] = (m < p.M && k < k_end) ? load_f(A, m * p.a_m + k * p.a_k) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < PB; ++q) {
      const int e = threadIdx.x + q * SIMT_THREADS;
      const int nn = e % TN, kk = e / TN;
      const int n = n0 + nn, k = k0 + kk;
      rb[q] = (n < p.N && k < k_end) ? load_f(B, k * p.b_k + n * p.b_n) : 0.f;
    }
  };
  if (k_begin < k_end) fetch(k_begin);
  for (int k0 = k_begin; k0 < k_end; k0 += TK) {
#pragma unroll
    for (int q = 0; q < PA; ++q) {
      const int e = threadIdx.x + q * SIMT_THREADS;
      As[e % TK][e / TK] = ra[q];
    }
#pragma unroll
    for (int q = 0; q < PB; ++q) {
      const int e = threadIdx.x + q * SIMT_THREADS;
      Bs[e / TN][e % TN] = rb[q];
    }
    __syncthreads();
    if (k0 + TK < k_end) fetch(k0 + TK);
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  const EpiArgs& e = p.epi;
  auto store = [&](int mm, int nn, float acc_v) {  // the epilogue of tile entry (mm, nn)
    const int m = m0 + mm, n = n0 + nn;
    if (m >= p.M || m >= e.row_limit || n >= p.N) return;
    const long long off =
        (static_cast<long long>(g) * e.row_g + m) * e.ld + static_cast<long long>(g) * e.col_g + n;
    float v = e.alpha * acc_v;
    if (e.X != nullptr) v += e.beta * e.X[off];
    if (e.Y != nullptr) v += e.gamma * e.Y[off];
    if (m == n) v += e.delta;
    if (e.out_f32 != nullptr) e.out_f32[off] = v;
    if (e.out_bf16 != nullptr) e.out_bf16[off] = __float2bfloat16_rn(v);
  };
  if (p.splits > 1) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) Ps[ty * 4 + i][tx * 4 + j] = acc[i][j];
    cluster_sync();  // every slice's partial tile is in its CTA's shared memory
    // rank s finalises tile entries [s chunk, (s + 1) chunk): all slices'
    // values of an entry are loaded at once, then added from rank 0 upwards
    // in order (the same sum whichever rank does it)
    const int chunk = TM * TN / p.splits;
    for (int idx = split * chunk + threadIdx.x; idx < (split + 1) * chunk; idx += SIMT_THREADS) {
      const int mm = idx / TN, nn = idx % TN;
      const uint32_t at = 4u * static_cast<uint32_t>(mm * (TN + 1) + nn);
      float v[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        v[r] = 0.f;
        if (r < p.splits)
          v[r] = r == split ? Ps[mm][nn]
                            : ld_cluster_f32(map_peer(smem_u32(&Ps[0][0]),
                                                      static_cast<uint32_t>(r)) + at);
      }
      float s = v[0];
#pragma unroll
      for (int r = 1; r < 8; ++r)
        if (r < p.splits) s += v[r];
      store(mm, nn, s);
    }
    cluster_sync();  // no CTA leaves while a peer still reads its tile
    return;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) store(ty * 4 + i, tx * 4 + j, acc[i][j]);
}

// The fp32 W0 product with the block-diagonal factors on both sides in one
// launch (blocks of b dividing 32, or b = 64, so that blocks tile the 32-wide
// K steps and the 64-column output tiles):
//   forward:  u = x P^T (per K step, as the A operand), C = v = u W0^T,
//             out = y = v R^T
//   backward: dv = dy R (A operand), C = du = dv W0, out = dx = du P
// Per K step the activation's rows (x or dy, the columns the step's blocks
// cover) and the left blocks' rows for the step's 32 columns are staged in
// shared memory and form the step's A tile there (a sum over the b columns
// of a block, in order), which then feeds the 64 x 64 tile product as in
// simt_gemm_kernel, K split over a cluster the same way.  After the split
// sums each finalising rank holds whole rows of C: it stores them if asked,
// and applies the right factor to them (the 64-column tile holds whole
// blocks).
struct SimtFusedArgs {
  int M, N, K, b, splits;
  const float* X;           // [M][K]: x or dy
  const float* L;           // left blocks [K/b][b][b]
  int l_trans;              // A[t][k] = sum_j X[t][g b + j] L_g[kl][j] (0) or L_g[j][kl] (1)
  const float* W;           // W0 as B(k, n) = W[k w_k + n w_n]
  long long w_k, w_n;
  const float* R;           // right blocks [N/b][b][b] (null: C only)
  int r_trans;              // out[t][n] = sum_j C[t][g b + j] R_g[nl][j] (0) or R_g[j][nl] (1)
  float* C;                 // [M][N] (null: not stored)
  float* out;               // [M][N]
};

constexpr int kFusedSmemFloats = TK * (TM + 4) + TK * (TN + 4) + 2 * TM * (TN + 1) +
                                 TM * (kFusedXW + 1) + TK * (kFusedXW + 1) + TN * (kFusedXW + 1);

// B: the block size (a template parameter, so that every staging loop has a
// fixed trip count and a thread's global loads of a step are all in flight
// before it stores any of them).
template <int B>
__global__ void __launch_bounds__(SIMT_THREADS) simt_fused_kernel(const SimtFusedArgs p) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ float fsm[];
  float (*As)[TM + 4] = reinterpret_cast<float (*)[TM + 4]>(fsm);
  float (*Bs)[TN + 4] = reinterpret_cast<float (*)[TN + 4]>(fsm + TK * (TM + 4));
  float (*Ps)[TN + 1] = reinterpret_cast<float (*)[TN + 1]>(fsm + TK * (TM + 4) + TK * (TN + 4));
  float (*Cs)[TN + 1] = Ps + TM;  // the finalised rows of C
  float (*Xs)[kFusedXW + 1] = reinterpret_cast<float (*)[kFusedXW + 1]>(Cs + TM);
  float (*Ls)[kFusedXW + 1] = Xs + TM;
  float (*Rs)[kFusedXW + 1] = Ls + TK;
  constexpr int XW = B >= TK ? B : TK;           // activation columns a K step reads
  constexpr int NX = TM * XW / SIMT_THREADS;     // per thread: activation values
  constexpr int NL = (TK * B + SIMT_THREADS - 1) / SIMT_THREADS;  // left block values
  constexpr int NW = TN * TK / SIMT_THREADS;     // W0 values
  constexpr int NR = (TN * B + SIMT_THREADS - 1) / SIMT_THREADS;  // right block values
  const int m0 = blockIdx.y * TM;
  const int split = p.splits > 1 ? static_cast<int>(blockIdx.x) % p.splits : 0;
  const int n0 = (p.splits > 1 ? static_cast<int>(blockIdx.x) / p.splits : blockIdx.x) * TN;
  const int kslice = ((p.K + p.splits * TK - 1) / (p.splits * TK)) * TK;
  const int k_begin = split * kslice;
  const int k_end = min(p.K, k_begin + kslice);
  const int tx = threadIdx.x % 16;  // n direction
  const int ty = threadIdx.x / 16;  // m direction

  // the right factor's rows for the tile's columns: loaded first, stored
  // after the first step's loads are in flight
  float rr[NR];
  if (p.R != nullptr) {
#pragma unroll
    for (int q = 0; q < NR; ++q) {
      const int e = threadIdx.x + q * SIMT_THREADS;
      const int nn = e / B, j = e - nn * B;
      const int n = n0 + nn;
      rr[q] = 0.f;
      if (e < TN * B && n < p.N) {
        const int blk = n / B, nl = n - blk * B;
        const float* Rb = p.R + static_cast<long long>(blk) * B * B;
        rr[q] = p.r_trans ? Rb[j * B + nl] : Rb[nl * B + j];
      }
    }
  }
  float acc[4][4] = {};
  bool r_stored = false;
  for (int k0 = k_begin; k0 < k_end; k0 += TK) {
    const int xb = B >= TK ? (k0 / B) * B : k0;  // the first activation column
    float rx[NX], rl[NL], rw[NW];
#pragma unroll
    for (int q = 0; q < NX; ++q) {
      const int e = threadIdx.x + q * SIMT_THREADS;
      const int mm = e / XW, c = e - mm * XW;
      const int m = m0 + mm, col = xb + c;
      rx[q] = (m < p.M && col < p.K) ? p.X[static_cast<long long>(m) * p.K + col] : 0.f;
    }
#pragma unroll
    for (int q = 0; q < NL; ++q) {
      const int e = threadIdx.x + q * SIMT_THREADS;
      const int kk = e / B, j = e - kk * B;
      const int k = k0 + kk;
      rl[q] = 0.f;
      if (e < TK * B && k < k_end) {
        const int blk = k / B, kl = k - blk * B;
        const float* Lb = p.L + static_cast<long long>(blk) * B * B;
        rl[q] = p.l_trans ? Lb[j * B + kl] : Lb[kl * B + j];
      }
    }
#pragma unroll
    for (int q = 0; q < NW; ++q) {
      const int e = threadIdx.x + q * SIMT_THREADS;
      const int nn = e % TN, kk = e / TN;
      const int n = n0 + nn, k = k0 + kk;
      rw[q] = (n < p.N && k < k_end) ? p.W[k * p.w_k + n * p.w_n] : 0.f;
    }
    if (p.R != nullptr && !r_stored) {
#pragma unroll
      for (int q = 0; q < NR; ++q) {
        const int e = threadIdx.x + q * SIMT_THREADS;
        if (e < TN * B) Rs[e / B][e % B] = rr[q];
      }
      r_stored = true;
    }
#pragma unroll
    for (int q = 0; q < NX; ++q) {
      const int e = threadIdx.x + q * SIMT_THREADS;
      Xs[e / XW][e % XW] = rx[q];
    }
#pragma unroll
    for (int q = 0; q < NL; ++q) {
      const int e = threadIdx.x + q * SIMT_THREADS;
      if (e < TK * B) Ls[e / B][e % B] = rl[q];
    }
#pragma unroll
    for (int q = 0; q < NW; ++q) {
      const int e = threadIdx.x + q * SIMT_THREADS;
      Bs[e / TN][e % TN] = rw[q];
    }
    __syncthreads();
    // the step's A tile: A[kk][m] = sum_j Xs[m][its block's column j] Ls[kk][j]
#pragma unroll
    for (int q = 0; q < TK * TM / SIMT_THREADS; ++q) {
      const int e = threadIdx.x + q * SIMT_THREADS;
      const int kk = e / TM, mm = e - kk * TM;
      const int xo = B >= TK ? 0 : (kk / B) * B;
      float s = 0.f;
#pragma unroll
      for (int j = 0; j < B; ++j) s = fmaf(Xs[mm][xo + j], Ls[kk][j], s);
      As[kk][mm] = s;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
  if (p.R != nullptr && !r_stored) {  // an empty K range
#pragma unroll
    for (int q = 0; q < NR; ++q) {
      const int e = threadIdx.x + q * SIMT_THREADS;
      if (e < TN * B) Rs[e / B][e % B] = rr[q];
    }
  }
  // the split sums: rank s finalises rows [s rows, (s + 1) rows) of C, all
  // slices' values of an entry loaded at once and added in rank order
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) Ps[ty * 4 + i][tx * 4 + j] = acc[i][j];
  if (p.splits > 1)
    cluster_sync();
  else
    __syncthreads();
  const int rows = TM / p.splits, r0 = split * rows;
  for (int idx = threadIdx.x; idx < rows * TN; idx += SIMT_THREADS) {
    const int mm = r0 + idx / TN, nn = idx % TN;
    const uint32_t at = 4u * static_cast<uint32_t>(mm * (TN + 1) + nn);
    float v[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      v[r] = 0.f;
      if (r < p.splits)
        v[r] = r == split ? Ps[mm][nn]
                          : ld_cluster_f32(map_peer(smem_u32(&Ps[0][0]), static_cast<uint32_t>(r)) +
                                           at);
    }
    float s = v[0];
#pragma unroll
    for (int r = 1; r < 8; ++r)
      if (r < p.splits) s += v[r];
    Cs[mm][nn] = s;
    const int m = m0 + mm, n = n0 + nn;
    if (p.C != nullptr && m < p.M && n < p.N) p.C[static_cast<long long>(m) * p.N + n] = s;
  }
  if (p.splits > 1) cluster_sync();  // no CTA leaves or reuses Ps while a peer reads it
  if (p.R == nullptr) return;
  __syncthreads();
  for (int idx = threadIdx.x; idx < rows * TN; idx += SIMT_THREADS) {
    const int mm = r0 + idx / TN, nn = idx % TN;
    const int m = m0 + mm, n = n0 + nn;
    if (m >= p.M || n >= p.N) continue;
    const int co = (nn / B) * B;  // the block's first column in the tile
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < B; ++j) s = fmaf(Cs[mm][co + j], Rs[nn][j], s);
    p.out[static_cast<long long>(m) * p.N + n] = s;
  }
}

// Position of Q[i][j] (i < j) in the row-by-row packed strict upper triangle.
__device__ __forceinline__ int packed_pos(int i, int j, int b) {
  return i * b - (i * (i + 1)) / 2 + (j - i - 1);
}

// Blocks of b <= 64 (fp32 arithmetic), one CTA per block and every matrix in
// shared memory, so the whole recursion is one launch instead of one per
// product.  Each product entry is a plain fmaf sum over t = 0 .. b-1.
//   build:   E = Q;  k times E <- 2Q + Q E;  R = I + E
//   adjoint: H = G^T (G = dL/dR);  P = Y = H;  k times P <- 2H + P Q,
//            Y <- P + Q Y;  D = Y = (dL/dQ)^T;  dtheta(i, j) = D[j][i] - D[i][j]
// (the reverse sweep of the build regrouped by Horner's rule on both sides
// of H: both recursions run forward and no power of Q is kept).
constexpr int kSmallMaxB = 64;

// Q from the packed strict upper triangle th.  With b x b = PER x blockDim.x
// (PER = 1, 4, 16), a thread's PER entries are loaded before any of them is
// stored; otherwise one entry at a time.
template <int PER>
__device__ __forceinline__ void small_load_q_per(const float* th, int b, float* Q) {
  float v[PER];
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int e = threadIdx.x + u * blockDim.x;
    const int i = e / b, j = e - (e / b) * b;
    v[u] = i < j ? th[packed_pos(i, j, b)] : (i > j ? -th[packed_pos(j, i, b)] : 0.f);
  }
#pragma unroll
  for (int u = 0; u < PER; ++u) Q[threadIdx.x + u * blockDim.x] = v[u];
}

__device__ __forceinline__ void small_load_q(const float* th, int b, float* Q) {
  const int bb = b * b;
  if (bb % blockDim.x == 0) {
    switch (bb / blockDim.x) {
      case 1: return small_load_q_per<1>(th, b, Q);
      case 4: return small_load_q_per<4>(th, b, Q);
      case 16: return small_load_q_per<16>(th, b, Q);
      default: break;
    }
  }
  for (int e = threadIdx.x; e < bb; e += blockDim.x) {
    const int i = e / b, j = e - (e / b) * b;
    Q[e] = i < j ? th[packed_pos(i, j, b)] : (i > j ? -th[packed_pos(j, i, b)] : 0.f);
  }
}

// out = xs X + Y + L R  (b x b, row-major; X, Y may be null; none of them
// aliases out).  When blockDim.x is a multiple of b and the b x b outputs
// are PER times blockDim.x, a thread's outputs (e, e + blockDim.x, ..) share
// one column j: R[t][j] is loaded once per t for all PER of them.  Every
// output is the same fmaf sum over t = 0 .. b-1 either way.
template <int PER>
__device__ __forceinline__ void small_mm_cols(int b, const float* L, const float* R,
                                              const float* X, float xs, const float* Y,
                                              float* out) {
  const int j = threadIdx.x % b, i0 = threadIdx.x / b, di = blockDim.x / b;
  float acc[PER];
#pragma unroll
  for (int r = 0; r < PER; ++r) acc[r] = 0.f;
  for (int t = 0; t < b; ++t) {
    const float rv = R[t * b + j];
#pragma unroll
    for (int r = 0; r < PER; ++r) acc[r] = fmaf(L[(i0 + r * di) * b + t], rv, acc[r]);
  }
#pragma unroll
  for (int r = 0; r < PER; ++r) {
    const int e = (i0 + r * di) * b + j;
    float v = acc[r];
    if (X != nullptr) v = xs * X[e] + v;
    if (Y != nullptr) v = Y[e] + v;
    out[e] = v;
  }
}

__device__ __forceinline__ void small_mm(int b, const float* L, const float* R, const float* X,
                                         float xs, const float* Y, float* out) {
  const int bb = b * b, nt = blockDim.x;
  if (nt % b == 0 && bb % nt == 0) {
    switch (bb / nt) {
      case 1: return small_mm_cols<1>(b, L, R, X, xs, Y, out);
      case 4: return small_mm_cols<4>(b, L, R, X, xs, Y, out);
      case 16: return small_mm_cols<16>(b, L, R, X, xs, Y, out);
      default: break;
    }
  }
  for (int e = threadIdx.x; e < bb; e += nt) {
    const int i = e / b, j = e - (e / b) * b;
    float acc = 0.f;
    for (int t = 0; t < b; ++t) acc = fmaf(L[i * b + t], R[t * b + j], acc);
    float v = acc;
    if (X != nullptr) v = xs * X[e] + v;
    if (Y != nullptr) v = Y[e] + v;
    out[e] = v;
  }
}

__global__ void __launch_bounds__(256) small_build_kernel(const float* __restrict__ theta, int b,
                                                          int k, float* __restrict__ out32,
                                                          __nv_bfloat16* __restrict__ out16) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ float small_smem[];
  const int bb = b * b;
  float* Q = small_smem;
  float* E = Q + bb;
  float* F = E + bb;
  const long long g = blockIdx.x;
  small_load_q(theta + g * (static_cast<long long>(b) * (b - 1) / 2), b, Q);
  __syncthreads();
  for (int e = threadIdx.x; e < bb; e += blockDim.x) E[e] = Q[e];
  __syncthreads();
  for (int it = 0; it < k; ++it) {
    small_mm(b, Q, E, Q, 2.f, nullptr, F);  // F = 2Q + Q E
    __syncthreads();
    float* t = E;
    E = F;
    F = t;
  }
  for (int e = threadIdx.x; e < bb; e += blockDim.x) {
    const int i = e / b, j = e - (e / b) * b;
    const float v = E[e] + (i == j ? 1.f : 0.f);
    if (out32 != nullptr) out32[g * bb + e] = v;
    if (out16 != nullptr) out16[g * bb + e] = __float2bfloat16_rn(v);
  }
}

__global__ void __launch_bounds__(256) small_adjoint_kernel(
    const float* __restrict__ theta_a, int n_a, const float* __restrict__ theta_b, int b, int k,
    const float* __restrict__ G, float* __restrict__ dtheta_a, float* __restrict__ dtheta_b) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ float small_smem[];
  const int bb = b * b;
  const long long m = static_cast<long long>(b) * (b - 1) / 2;
  float* Q = small_smem;
  float* H = Q + bb;
  float* P = H + bb;
  float* Y = P + bb;
  float* P2 = Y + bb;
  float* Y2 = P2 + bb;
  const int g = blockIdx.x;
  const bool side_b = g >= n_a;
  const long long lg = side_b ? g - n_a : g;
  small_load_q((side_b ? theta_b : theta_a) + lg * m, b, Q);
  const float* Gg = G + static_cast<long long>(g) * bb;
  // H = G^T (and the first P and Y); a thread's PER entries loaded before
  // any is stored when b x b = PER x blockDim.x
  auto load_h = [&](auto per_c) {
    constexpr int PER = decltype(per_c)::value;
    float v[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int e = threadIdx.x + u * blockDim.x;
      const int i = e / b, j = e - (e / b) * b;
      v[u] = Gg[j * b + i];
    }
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int e = threadIdx.x + u * blockDim.x;
      H[e] = v[u];
      P[e] = v[u];
      Y[e] = v[u];
    }
  };
  if (bb == 4 * static_cast<int>(blockDim.x)) {
    load_h(std::integral_constant<int, 4>{});
  } else if (bb == 16 * static_cast<int>(blockDim.x)) {
    load_h(std::integral_constant<int, 16>{});
  } else {
    for (int e = threadIdx.x; e < bb; e += blockDim.x) {
      const int i = e / b, j = e - (e / b) * b;
      const float h = Gg[j * b + i];
      H[e] = h;
      P[e] = h;
      Y[e] = h;
    }
  }
  __syncthreads();
  for (int it = 0; it < k; ++it) {
    small_mm(b, P, Q, H, 2.f, nullptr, P2);  // P2 = 2H + P Q
    __syncthreads();
    small_mm(b, Q, Y, nullptr, 0.f, P2, Y2);  // Y2 = P2 + Q Y
    __syncthreads();
    float* t = P;
    P = P2;
    P2 = t;
    t = Y;
    Y = Y2;
    Y2 = t;
  }
  float* out = (side_b ? dtheta_b : dtheta_a) + lg * m;
  for (int e = threadIdx.x; e < bb; e += blockDim.x) {
    const int i = e / b, j = e - (e / b) * b;
    if (i < j) out[packed_pos(i, j, b)] = Y[j * b + i] - Y[i * b + j];
  }
}

// Token sums of fp32 blocks of b <= 64: G[g][m][n] = sum_t A[t][g b + m] B[t][g b + n]
// for the d / b blocks g (one side's block gradients).  One cluster of
// `splits` CTAs per block, each CTA a contiguous token range staged 64
// tokens at a time in shared memory (a token's b-wide pieces of A and B are
// consecutive words); each rank then finalises a share of the b x b sums,
// adding the CTAs' partial values in rank order (a fixed summation order,
// no scratch, no atomics).
constexpr int kOuterTC = 64;                                    // tokens per staged chunk
constexpr int kOuterPer = kSmallMaxB * kSmallMaxB / 256;        // outputs per thread

// One launch may cover two sides (the P and R blocks of a layer): blocks
// g < n_a belong to side 0, the rest to side 1.
struct OuterSides {
  const float* A[2];
  const float* B[2];
  float* G[2];
  int d[2];
  int n_a;
};

__global__ void __launch_bounds__(256) small_outer_kernel(const OuterSides sides, int b,
                                                          long long T, int splits) {
  pdl_wait();
  pdl_trigger();
  __shared__ float As[kOuterTC][kSmallMaxB];
  __shared__ float Bs[kOuterTC][kSmallMaxB];
  __shared__ float Ps[kSmallMaxB * kSmallMaxB];  // this CTA's partial sums (splits > 1)
  const int side = static_cast<int>(blockIdx.y) >= sides.n_a ? 1 : 0;
  const int g = static_cast<int>(blockIdx.y) - (side ? sides.n_a : 0);
  const float* __restrict__ A = sides.A[side];
  const float* __restrict__ B = sides.B[side];
  float* __restrict__ G = sides.G[side];
  const int d = sides.d[side];
  const int split = blockIdx.x;  // the rank in the block's cluster
  const long long per = (T + splits - 1) / splits;
  const long long t0 = split * per;
  const long long t1 = t0 + per < T ? t0 + per : T;
  const int bb = b * b;
  const long long col0 = static_cast<long long>(g) * b;
  float acc[kOuterPer];
#pragma unroll
  for (int i = 0; i < kOuterPer; ++i) acc[i] = 0.f;
  for (long long c = t0; c < t1; c += kOuterTC) {
    const long long left = t1 - c;
    const int nt = left < kOuterTC ? static_cast<int>(left) : kOuterTC;
    if ((b & 3) == 0) {
      // 16-byte pieces (b, d and the block offset are multiples of 4 floats;
      // the activations are 16-byte aligned): every load of the thread is
      // issued before any of them is stored (at most 4 pieces per operand)
      const int q4 = b >> 2, total = kOuterTC * q4;
      float4 av[4], bv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = threadIdx.x + u * 256;
        av[u] = bv[u] = make_float4(0.f, 0.f, 0.f, 0.f);  // tokens past the range: zeros
        if (e < total) {
          const int tt = e / q4, j4 = e - tt * q4;
          if (tt < nt) {
            const long long off = (c + tt) * d + col0 + 4 * j4;
            av[u] = *reinterpret_cast<const float4*>(A + off);
            bv[u] = *reinterpret_cast<const float4*>(B + off);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int e = threadIdx.x + u * 256;
        if (e < total) {
          const int tt = e / q4, j = 4 * (e - tt * q4);
          As[tt][j] = av[u].x;
          As[tt][j + 1] = av[u].y;
          As[tt][j + 2] = av[u].z;
          As[tt][j + 3] = av[u].w;
          Bs[tt][j] = bv[u].x;
          Bs[tt][j + 1] = bv[u].y;
          Bs[tt][j + 2] = bv[u].z;
          Bs[tt][j + 3] = bv[u].w;
        }
      }
    } else {
      for (int e = threadIdx.x; e < kOuterTC * b; e += blockDim.x) {
        const int tt = e / b, j = e - tt * b;
        float av = 0.f, bv = 0.f;  // tokens past the range: zeros, which add nothing
        if (tt < nt) {
          const long long off = (c + tt) * d + col0 + j;
          av = A[off];
          bv = B[off];
        }
        As[tt][j] = av;
        Bs[tt][j] = bv;
      }
    }
    __syncthreads();
    // a thread's outputs share column n when 256 % b == 0: Bs[tt][n] loaded
    // once per token for all of them
    auto cols = [&](auto per_c) {
      constexpr int PER = decltype(per_c)::value;
      const int n = threadIdx.x % b, m0 = threadIdx.x / b, dm = 256 / b;
      for (int tt = 0; tt < kOuterTC; ++tt) {
        const float bv = Bs[tt][n];
#pragma unroll
        for (int i = 0; i < PER; ++i) acc[i] = fmaf(As[tt][m0 + i * dm], bv, acc[i]);
      }
    };
    if (bb == 4096) {
      cols(std::integral_constant<int, 16>{});
    } else if (bb == 1024) {
      cols(std::integral_constant<int, 4>{});
    } else if (bb == 256) {
      cols(std::integral_constant<int, 1>{});
    } else {
#pragma unroll
      for (int i = 0; i < kOuterPer; ++i) {
        const int o = threadIdx.x + i * 256;
        if (o < bb) {
          const int m = o / b, n = o - m * b;
          float s = acc[i];
#pragma unroll 8
          for (int tt = 0; tt < kOuterTC; ++tt) s = fmaf(As[tt][m], Bs[tt][n], s);
          acc[i] = s;
        }
      }
    }
    __syncthreads();
  }
  if (splits > 1) {
#pragma unroll
    for (int i = 0; i < kOuterPer; ++i) {
      const int o = threadIdx.x + i * 256;
      if (o < bb) Ps[o] = acc[i];
    }
    cluster_sync();  // every CTA's partial sums are in its shared memory
    // rank s finalises outputs [s chunk, (s + 1) chunk): all ranks' values of
    // an output are loaded at once, then added from rank 0 upwards in order
    const int chunk = (bb + splits - 1) / splits;
    const int o_end = min(bb, (split + 1) * chunk);
    for (int o = split * chunk + threadIdx.x; o < o_end; o += blockDim.x) {
      float v[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        v[r] = 0.f;
        if (r < splits)
          v[r] = r == split ? Ps[o]
                            : ld_cluster_f32(map_peer(smem_u32(Ps), static_cast<uint32_t>(r)) +
                                             4u * static_cast<uint32_t>(o));
      }
      float s = v[0];
#pragma unroll
      for (int r = 1; r < 8; ++r)
        if (r < splits) s += v[r];
      G[static_cast<long long>(g) * bb + o] = s;
    }
    cluster_sync();  // no CTA leaves while a peer still reads its partial sums
    return;
  }
#pragma unroll
  for (int i = 0; i < kOuterPer; ++i) {
    const int o = threadIdx.x + i * 256;
    if (o < bb) G[static_cast<long long>(g) * bb + o] = acc[i];
  }
}

// Index arithmetic below is 32-bit: the host guarantees n * b * b < 2^31.
// Blocks [0, n_a) come from theta_a, blocks [n_a, n_a + n_b) from theta_b.
__global__ void unpack_kernel(const float* __restrict__ theta_a, int n_a,
                              const float* __restrict__ theta_b, int b, int total,
                              float* __restrict__ q32, __nv_bfloat16* __restrict__ q16) {
  pdl_wait();
  pdl_trigger();
  const int bb = b * b;
  const int m = b * (b - 1) / 2;
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += gridDim.x * blockDim.x) {
    const int g = idx / bb;
    const int rem = idx - g * bb;
    const int i = rem / b;
    const int j = rem - i * b;
    const float* th = g < n_a ? theta_a + g * m : theta_b + (g - n_a) * m;
    float v = 0.f;
    if (i < j) v = th[packed_pos(i, j, b)];
    else if (i > j) v = -th[packed_pos(j, i, b)];
    if (q32 != nullptr) q32[idx] = v;
    if (q16 != nullptr) q16[idx] = __float2bfloat16_rn(v);
  }
}

__global__ void identity_plus_kernel(const float* __restrict__ q, int b, int total,
                                     float* __restrict__ o32, __nv_bfloat16* __restrict__ o16) {
  pdl_wait();
  pdl_trigger();
  const int bb = b * b;
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += gridDim.x * blockDim.x) {
    const int rem = idx % bb;
    const int i = rem / b;
    const int j = rem - i * b;
    const float v = q[idx] + (i == j ? 1.f : 0.f);
    if (o32 != nullptr) o32[idx] = v;
    if (o16 != nullptr) o16[idx] = __float2bfloat16_rn(v);
  }
}

// One 16-byte vector (8 columns) per thread: b is a multiple of 8, so the
// vector lies in one block column and is either a copy of 8 block entries
// (16-byte aligned: b * b and b are multiples of 8) or zero.  total8 counts
// vectors.
__global__ void expand_superblocks_kernel(const __nv_bfloat16* __restrict__ blocks, int n, int b,
                                          int S, int total8, __nv_bfloat16* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  const int per = S / b;
  const int vrow = S / 8;  // vectors per superblock row
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < total8;
       idx += gridDim.x * blockDim.x) {
    const int c = 8 * (idx % vrow);
    const int r = (idx / vrow) % S;
    const int sb = idx / (vrow * S);
    const int gblk = sb * per + r / b;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (r / b == c / b && gblk < n)
      v = *reinterpret_cast<const uint4*>(blocks + (static_cast<long long>(gblk) * b + (r % b)) * b +
                                          (c % b));
    reinterpret_cast<uint4*>(out)[idx] = v;
  }
}

// out[g] (g < n) = sum over splits of the diagonal b-block of superblock
// g / (S/b) in part [splits][nsb][S][S].
__global__ void reduce_extract_kernel(const float* __restrict__ part, int splits, int n, int b,
                                      int S, int total, float* __restrict__ o32,
                                      __nv_bfloat16* __restrict__ o16) {
  pdl_wait();
  pdl_trigger();
  const int per = S / b;
  const int nsb = (n + per - 1) / per;
  const long long split_stride = static_cast<long long>(nsb) * S * S;
  const int bb = b * b;
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += gridDim.x * blockDim.x) {
    const int g = idx / bb;
    const int rem = idx - g * bb;
    const int i = rem / b;
    const int j = rem - i * b;
    const int sb = g / per;
    const int off = (g - sb * per) * b;
    const long long src = (static_cast<long long>(sb) * S + off + i) * S + off + j;
    float v = 0.f;
    for (int s = 0; s < splits; ++s) v += part[s * split_stride + src];
    if (o32 != nullptr) o32[idx] = v;
    if (o16 != nullptr) o16[idx] = __float2bfloat16_rn(v);
  }
}

// dtheta[g][idx(i,j)] = M[g][i][j] - M[g][j][i], M = A (+ B): one thread per
// (g, i, j) with i < j; blocks [0, n_a) go to dtheta_a, the rest to dtheta_b.
__global__ void pack_skew_kernel(const float* __restrict__ A, const float* __restrict__ B, int n_a,
                                 int b, int total, float* __restrict__ dtheta_a,
                                 float* __restrict__ dtheta_b) {
  pdl_wait();
  pdl_trigger();
  const int m = b * (b - 1) / 2;
  const int bb = b * b;
  for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += gridDim.x * blockDim.x) {
    const int g = idx / bb;
    const int rem = idx - g * bb;
    const int i = rem / b;
    const int j = rem - i * b;
    if (i >= j) continue;
    const int ji = g * bb + j * b + i;
    float v = A[idx] - A[ji];
    if (B != nullptr) v += B[idx] - B[ji];
    if (g < n_a) dtheta_a[g * m + packed_pos(i, j, b)] = v;
    else dtheta_b[(g - n_a) * m + packed_pos(i, j, b)] = v;
  }
}

__global__ void f32_to_bf16_kernel(const float* __restrict__ in, long long count,
                                   __nv_bfloat16* __restrict__ out) {
  pdl_wait();
  pdl_trigger();
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < count;
       idx += static_cast<long long>(gridDim.x) * blockDim.x)
    out[idx] = __float2bfloat16_rn(in[idx]);
}

// --------------------------------------------------- 32 x 32 tile kernels
// One CTA of 256 threads per 32 x 32 tile (ti, tj) of one b x b block; thread
// (r, c4) owns row r, columns c4 .. c4+3 of the tile (16-byte fp32 / 8-byte
// bf16 accesses).  The transposed half of a skew matrix goes through a
// shared-memory tile, so it is read and written row-wise as well.

constexpr int TT = 32;

__device__ __forceinline__ void store_bf16x4(__nv_bfloat16* dst, float a, float b, float c,
                                             float d) {
  const __nv_bfloat162 lo = __floats2bfloat162_rn(a, b);
  const __nv_bfloat162 hi = __floats2bfloat162_rn(c, d);
  uint2 w;
  w.x = *reinterpret_cast<const uint32_t*>(&lo);
  w.y = *reinterpret_cast<const uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(dst) = w;
}

// bf16 value, bf16 remainder and twice the bf16 value of four entries
__device__ __forceinline__ void store_hi_lo(__nv_bfloat16* hi, __nv_bfloat16* lo,
                                            __nv_bfloat16* x2, const float* q) {
  float h[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) h[e] = __bfloat162float(__float2bfloat16_rn(q[e]));
  store_bf16x4(hi, h[0], h[1], h[2], h[3]);
  if (lo != nullptr) store_bf16x4(lo, q[0] - h[0], q[1] - h[1], q[2] - h[2], q[3] - h[3]);
  if (x2 != nullptr) store_bf16x4(x2, 2.f * h[0], 2.f * h[1], 2.f * h[2], 2.f * h[3]);
}

// Q from theta for the tile pair (ti, tj), (tj, ti) with ti <= tj; writes
// the bf16 value (hi) and optionally the bf16 remainder (lo) of each entry.
__device__ __forceinline__ void unpack_tile_pair(const float* __restrict__ th, int b, int ti,
                                                 int tj, __nv_bfloat16* __restrict__ hi,
                                                 __nv_bfloat16* __restrict__ lo,
                                                 __nv_bfloat16* __restrict__ x2,
                                                 float (*tile)[TT + 1]) {
  const int tid = threadIdx.x;
  for (int e = tid; e < TT * TT; e += 256) {  // upper entries (i < j) of tile (ti, tj)
    const int rr = e / TT, cc = e % TT;
    const int i = ti * TT + rr, j = tj * TT + cc;
    tile[rr][cc] = i < j ? th[packed_pos(i, j, b)] : 0.f;
  }
  __syncthreads();
  const int r = tid >> 3, c4 = (tid & 7) * 4;
  // tile (ti, tj): Q[i][j] = theta (i < j), -theta[j][i] (below the diagonal), 0
  float q[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int c = c4 + e;
    q[e] = (ti == tj && r > c) ? -tile[c][r] : tile[r][c];
  }
  const long long o = static_cast<long long>(ti * TT + r) * b + tj * TT + c4;
  store_hi_lo(hi + o, lo != nullptr ? lo + o : nullptr, x2 != nullptr ? x2 + o : nullptr, q);
  if (ti != tj) {  // mirrored tile (tj, ti): Q[j'][i'] = -theta[i'][j']
#pragma unroll
    for (int e = 0; e < 4; ++e) q[e] = -tile[c4 + e][r];
    const long long o2 = static_cast<long long>(tj * TT + r) * b + ti * TT + c4;
    store_hi_lo(hi + o2, lo != nullptr ? lo + o2 : nullptr, x2 != nullptr ? x2 + o2 : nullptr,
                q);
  }
}

// Tile pair k (k < t(t+1)/2) of a t x t tiling: tiles (ti, tj) and (tj, ti), ti <= tj.
__device__ __forceinline__ void tile_pair(int k, int t, int& ti, int& tj) {
  ti = 0;
  while (k >= t - ti) {
    k -= t - ti;
    ++ti;
  }
  tj = ti + k;
}

// grid (tile pairs per block, n_a + n_b), 256 threads; for tiles (ti, tj) and
// (tj, ti) of block g:
//   Q (bf16, plus lo if q_lo, plus 2Q if q_x2) from theta,
//   2I into two_i for block 0,
//   F = sum over splits of the diagonal b-block of the partials (if f16).
__global__ void __launch_bounds__(256) prep_tiles_kernel(PrepTilesArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ float tile[TT][TT + 1];
  const int t = a.b / TT;
  int ti, tj;
  tile_pair(blockIdx.x, t, ti, tj);
  const int g = blockIdx.y;
  const long long bb = static_cast<long long>(a.b) * a.b;
  const int m = a.b * (a.b - 1) / 2;
  const bool side_a = g < a.n_a;
  const int gl = side_a ? g : g - a.n_a;
  const int tid = threadIdx.x;
  const int r = tid >> 3, c4 = (tid & 7) * 4;
  if (a.zero_words != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && tid < a.n_zero_words)
    a.zero_words[tid] = 0u;
  const int ntiles = ti == tj ? 1 : 2;
  if (a.f16 != nullptr) {
    const int per = a.S / a.b;
    const int sb = gl / per;
    const int off = (gl - sb * per) * a.b;
    const float* part = side_a ? a.part_a : a.part_b;
    const int splits = side_a ? a.splits_a : a.splits_b;
    const long long stride = static_cast<long long>(side_a ? a.nsb_a : a.nsb_b) * a.S * a.S;
    for (int q = 0; q < ntiles; ++q) {
      const int i = (q == 0 ? ti : tj) * TT + r, j0 = (q == 0 ? tj : ti) * TT + c4;
      const long long src = (static_cast<long long>(sb) * a.S + off + i) * a.S + off + j0;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int s = 0; s < splits; ++s) {
        const float4 w = *reinterpret_cast<const float4*>(part + s * stride + src);
        v.x += w.x;
        v.y += w.y;
        v.z += w.z;
        v.w += w.w;
      }
      const long long o = g * bb + static_cast<long long>(i) * a.b + j0;
      store_bf16x4(a.f16 + o, v.x, v.y, v.z, v.w);
      if (a.f32 != nullptr) *reinterpret_cast<float4*>(a.f32 + o) = v;
    }
  }
  if (g == 0 && a.two_i != nullptr) {
    for (int q = 0; q < ntiles; ++q) {
      const int i = (q == 0 ? ti : tj) * TT + r, j0 = (q == 0 ? tj : ti) * TT + c4;
      store_bf16x4(a.two_i + static_cast<long long>(i) * a.b + j0, i == j0 ? 2.f : 0.f,
                   i == j0 + 1 ? 2.f : 0.f, i == j0 + 2 ? 2.f : 0.f, i == j0 + 3 ? 2.f : 0.f);
    }
  }
  if (a.q_hi != nullptr) {
    const float* th = side_a ? a.theta_a + static_cast<long long>(gl) * m
                             : a.theta_b + static_cast<long long>(gl) * m;
    unpack_tile_pair(th, a.b, ti, tj, a.q_hi + g * bb,
                     a.q_lo != nullptr ? a.q_lo + g * bb : nullptr,
                     a.q_x2 != nullptr ? a.q_x2 + g * bb : nullptr, tile);
  }
}

// dtheta[g][idx(i,j)] = sign * (D[g][i][j] - D[g][j][i]) for the i < j entries of
// tile (ti, tj), ti <= tj; grid (tile pairs per block, n_a + n_b), 256 threads.
__global__ void __launch_bounds__(256) pack_tiles_kernel(const float* __restrict__ D, float sign,
                                                         int n_a, int b,
                                                         float* __restrict__ dtheta_a,
                                                         float* __restrict__ dtheta_b) {
  pdl_wait();
  pdl_trigger();
  __shared__ float tile[TT][TT + 1];
  const int t = b / TT;
  int ti, tj;
  tile_pair(blockIdx.x, t, ti, tj);
  const int g = blockIdx.y;
  const long long base = static_cast<long long>(g) * b * b;
  const int m = b * (b - 1) / 2;
  const int tid = threadIdx.x;
  const int r = tid >> 3, c4 = (tid & 7) * 4;
  {  // D[j][i] for the tile: rows of tile (tj, ti)
    const float4 w =
        *reinterpret_cast<const float4*>(D + base + static_cast<long long>(tj * TT + r) * b +
                                         ti * TT + c4);
    tile[r][c4] = w.x;
    tile[r][c4 + 1] = w.y;
    tile[r][c4 + 2] = w.z;
    tile[r][c4 + 3] = w.w;
  }
  __syncthreads();
  float* out = g < n_a ? dtheta_a + static_cast<long long>(g) * m
                       : dtheta_b + static_cast<long long>(g - n_a) * m;
  const int i = ti * TT + r, j0 = tj * TT + c4;
  const float4 dij =
      *reinterpret_cast<const float4*>(D + base + static_cast<long long>(i) * b + j0);
  const float d4[4] = {dij.x, dij.y, dij.z, dij.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int j = j0 + e;
    if (i < j) out[packed_pos(i, j, b)] = sign * (d4[e] - tile[c4 + e][r]);
  }
}

// out[r][i] = in[row_map ? row_map[r] : r][col_map[i]] for r < rows, i < d.
// A CTA takes groups of R rows (R = 8 bytes / element: 4 bf16 or 2 fp32
// rows) in turn and writes them into a shared-memory table interleaved, one
// 8-byte entry per column holding that column of all R rows; the gather
// then reads 8-byte entries at the mapped columns, so one random
// shared-memory read serves R outputs, and assembles each row's 16 bytes of
// consecutive outputs.  Table order: the entry of column c sits at
// (c % V) * (d / V) + c / V (V columns per 16-byte vector), so a warp's
// stores of entries are consecutive 8-byte words; bf16 entries and output
// words are assembled by byte permutes.  A thread serves the same output
// vectors in every group and keeps the table positions of its first few
// vectors in registers.  Map entries outside [0, d) (or [0, in_rows)) are
// not followed: the output gets 0 and the status word POETX_ERR_INVALID_ARG.
//
// Two kernels move the rows:
//  - permute_bulk_kernel (rows of up to 9556 features, where two staged
//    groups and the table fit in shared memory): 1-D bulk copies bring a
//    group's source rows into one of two stages, all threads interleave the
//    stage into the table (after which the stage takes the copies of the
//    group two ahead), then gather and write the permuted rows with 16-byte
//    stores.  No thread waits on a global load, so the bytes in flight are
//    not bounded by registers.
//  - permute_rows_kernel (wider rows): producer warps read the source rows
//    with 16-byte loads straight into the table, consumer warps gather and
//    store with 16-byte stores; with two tables (NBUF = 2, when 16 d bytes
//    fit) the producers fill one while the consumers drain the other, and
//    named barriers hand the tables over.
constexpr int kPermRoleThreads = 128;  // producers, and as many consumers
constexpr int kPermThreads = 2 * kPermRoleThreads;
constexpr int kPermBulkThreads = 512;
constexpr size_t kPermSmemMax = 224 * 1024;

// The source rows of the group of R rows starting at r0 (-1: none, the
// output row is 0); returns whether a row-map entry was out of range.
template <int R>
__device__ __forceinline__ bool perm_group_sources(long long r0, long long rows,
                                                   const int* __restrict__ row_map,
                                                   long long in_rows, long long (&src)[R]) {
  bool bad = false;
#pragma unroll
  for (int q = 0; q < R; ++q) {
    const long long r = r0 + q;
    src[q] = -1;
    if (r < rows) {
      src[q] = r;
      if (row_map != nullptr) {
        const int m = row_map[r];
        src[q] = (m >= 0 && m < in_rows) ? m : -1;
        bad |= src[q] < 0;
      }
    }
  }
  return bad;
}

// Table entries of 16-byte source vector v of the R rows (wd[q] = row q's
// four words): column V v + e goes to position e * nv + v.
template <typename T>
__device__ __forceinline__ void perm_store_entries(uint2* ent, int nv, int v,
                                                   const uint32_t (&wd)[8 / sizeof(T)][4]) {
  constexpr int V = 16 / sizeof(T);
#pragma unroll
  for (int e = 0; e < V; ++e) {
    uint2 entry;
    if constexpr (sizeof(T) == 2) {  // column 8v + e: halves e % 2 of word e / 2
      const uint32_t sel = (e & 1) ? 0x7632u : 0x5410u;
      entry.x = __byte_perm(wd[0][e >> 1], wd[1][e >> 1], sel);
      entry.y = __byte_perm(wd[2][e >> 1], wd[3][e >> 1], sel);
    } else {
      entry.x = wd[0][e];
      entry.y = wd[1][e];
    }
    ent[e * nv + v] = entry;
  }
}

// Table positions of the map entries of output vector v, two 16-bit
// positions per word (0xffff: the entry is out of range, the output 0);
// returns whether any entry was out of range.
template <typename T>
__device__ __forceinline__ bool perm_table_positions(const int* __restrict__ col_map, int v, int d,
                                                     int nv, uint32_t (&pos)[8 / sizeof(T)]) {
  constexpr int V = 16 / sizeof(T);
  const int4* c4 = reinterpret_cast<const int4*>(col_map) + v * (V / 4);
  bool bad = false;
#pragma unroll
  for (int i = 0; i < V / 2; ++i) pos[i] = 0u;
#pragma unroll
  for (int qv = 0; qv < V / 4; ++qv) {
    const int4 c = c4[qv];
    const int cs[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int e = 4 * qv + t;
      const bool ok = cs[t] >= 0 && cs[t] < d;
      bad |= !ok;
      const uint32_t at = ok ? static_cast<uint32_t>((cs[t] & (V - 1)) * nv + cs[t] / V) : 0xffffu;
      pos[e >> 1] |= at << (16 * (e & 1));
    }
  }
  return bad;
}

// Output vector of the R rows from the entries at the table positions pos:
// o[q] = row q's four words.
template <typename T>
__device__ __forceinline__ void perm_gather(const uint2* ent, const uint32_t (&pos)[8 / sizeof(T)],
                                            uint32_t (&o)[8 / sizeof(T)][4]) {
  constexpr int V = 16 / sizeof(T);
  uint2 u[V];
#pragma unroll
  for (int e = 0; e < V; ++e) {
    const uint32_t at = (pos[e >> 1] >> (16 * (e & 1))) & 0xffffu;
    u[e] = at != 0xffffu ? ent[at] : make_uint2(0u, 0u);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (sizeof(T) == 2) {  // output word i: columns 2i, 2i + 1 of each row
      o[0][i] = __byte_perm(u[2 * i].x, u[2 * i + 1].x, 0x5410u);
      o[1][i] = __byte_perm(u[2 * i].x, u[2 * i + 1].x, 0x7632u);
      o[2][i] = __byte_perm(u[2 * i].y, u[2 * i + 1].y, 0x5410u);
      o[3][i] = __byte_perm(u[2 * i].y, u[2 * i + 1].y, 0x7632u);
    } else {
      o[0][i] = u[i].x;
      o[1][i] = u[i].y;
    }
  }
}

template <typename T, int NBUF>
__global__ void __launch_bounds__(kPermThreads, 3)
    permute_rows_kernel(const T* __restrict__ in, long long in_rows,
                        const int* __restrict__ row_map, const int* __restrict__ col_map,
                        T* __restrict__ out, long long rows, int d, int* status) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) unsigned char row_smem[];
  constexpr int V = 16 / sizeof(T);  // elements per 16-byte vector
  constexpr int R = 8 / sizeof(T);   // rows per group: one 8-byte entry per column
  constexpr int U = 8 / R;           // vectors of each row in flight per producer thread
  constexpr int KR = 4;              // vectors whose table positions a consumer keeps
  const int nv = d / V;
  const long long groups = (rows + R - 1) / R;
  const bool producer = threadIdx.x < kPermRoleThreads;
  const int tid = threadIdx.x % kPermRoleThreads;
  // this CTA's groups: blockIdx.x + n * gridDim.x, n < count
  const long long count =
      blockIdx.x < groups ? (groups - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;

  // named barriers 1 + b: table b is full; 1 + NBUF + b: table b is free
  // (immediate ids: a register id would reserve all sixteen barriers)
  auto bar_sync = [](int id) {
    switch (id) {
      case 1: asm volatile("bar.sync 1, %0;" ::"n"(kPermThreads) : "memory"); break;
      case 2: asm volatile("bar.sync 2, %0;" ::"n"(kPermThreads) : "memory"); break;
      case 3: asm volatile("bar.sync 3, %0;" ::"n"(kPermThreads) : "memory"); break;
      default: asm volatile("bar.sync 4, %0;" ::"n"(kPermThreads) : "memory"); break;
    }
  };
  auto bar_arrive = [](int id) {
    switch (id) {
      case 1: asm volatile("bar.arrive 1, %0;" ::"n"(kPermThreads) : "memory"); break;
      case 2: asm volatile("bar.arrive 2, %0;" ::"n"(kPermThreads) : "memory"); break;
      case 3: asm volatile("bar.arrive 3, %0;" ::"n"(kPermThreads) : "memory"); break;
      default: asm volatile("bar.arrive 4, %0;" ::"n"(kPermThreads) : "memory"); break;
    }
  };

  if (producer) {
    for (long long n = 0; n < count; ++n) {
      const int buf = static_cast<int>(n % NBUF);
      uint2* ent = reinterpret_cast<uint2*>(row_smem) + static_cast<size_t>(buf) * d;
      const long long r0 = (blockIdx.x + n * gridDim.x) * R;
      long long src[R];
      if (perm_group_sources<R>(r0, rows, row_map, in_rows, src) && tid == 0)
        atomicCAS(status, 0, 1);
      if (n >= NBUF) bar_sync(1 + NBUF + buf);  // the consumers are done with this table
      // interleave (missing rows: 0), U vectors of each row in flight
      for (int v0 = tid; v0 < nv; v0 += U * kPermRoleThreads) {
        uint4 w[U][R];
#pragma unroll
        for (int k = 0; k < U; ++k) {
          const int v = v0 + k * kPermRoleThreads;
#pragma unroll
          for (int q = 0; q < R; ++q) {
            w[k][q] = make_uint4(0u, 0u, 0u, 0u);
            if (v < nv && src[q] >= 0) w[k][q] = reinterpret_cast<const uint4*>(in + src[q] * d)[v];
          }
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
          const int v = v0 + k * kPermRoleThreads;
          if (v >= nv) break;
          uint32_t wd[R][4];
#pragma unroll
          for (int q = 0; q < R; ++q) {
            wd[q][0] = w[k][q].x;
            wd[q][1] = w[k][q].y;
            wd[q][2] = w[k][q].z;
            wd[q][3] = w[k][q].w;
          }
          perm_store_entries<T>(ent, nv, v, wd);
        }
      }
      bar_arrive(1 + buf);  // table full
    }
  } else {
    uint32_t pos_r[KR][V / 2];
    bool bad_cols = false;
#pragma unroll
    for (int k = 0; k < KR; ++k) {
      const int v = tid + k * kPermRoleThreads;
#pragma unroll
      for (int i = 0; i < V / 2; ++i) pos_r[k][i] = 0xffffffffu;
      if (v < nv) bad_cols |= perm_table_positions<T>(col_map, v, d, nv, pos_r[k]);
    }
    if (bad_cols && count > 0) atomicCAS(status, 0, 1);
    for (long long n = 0; n < count; ++n) {
      const int buf = static_cast<int>(n % NBUF);
      const uint2* ent = reinterpret_cast<const uint2*>(row_smem) + static_cast<size_t>(buf) * d;
      const long long r0 = (blockIdx.x + n * gridDim.x) * R;
      long long src[R];
      perm_group_sources<R>(r0, rows, row_map, in_rows, src);
      bar_sync(1 + buf);  // the producers have filled this table
      auto gather_store = [&](int v, const uint32_t (&pos)[V / 2]) {
        uint32_t o[R][4];
        perm_gather<T>(ent, pos, o);
#pragma unroll
        for (int q = 0; q < R; ++q) {
          if (r0 + q < rows) {
            uint4 val = make_uint4(o[q][0], o[q][1], o[q][2], o[q][3]);
            if (src[q] < 0) val = make_uint4(0u, 0u, 0u, 0u);
            reinterpret_cast<uint4*>(out + (r0 + q) * d)[v] = val;
          }
        }
      };
#pragma unroll
      for (int k = 0; k < KR; ++k) {
        const int v = tid + k * kPermRoleThreads;
        if (v < nv) gather_store(v, pos_r[k]);
      }
      for (int v = tid + KR * kPermRoleThreads; v < nv; v += kPermRoleThreads) {
        uint32_t pos[V / 2];
        if (perm_table_positions<T>(col_map, v, d, nv, pos)) atomicCAS(status, 0, 1);
        gather_store(v, pos);
      }
      if (n + NBUF < count) bar_arrive(1 + NBUF + buf);  // table free for group n + NBUF
    }
  }
}

// Shared memory of permute_bulk_kernel: two stages and the table (8 d bytes
// each), two mbarriers and the abort flag.
__host__ __device__ constexpr size_t perm_bulk_smem(int d) {
  return 3 * static_cast<size_t>(d) * 8 + 32;
}

template <typename T>
__global__ void __launch_bounds__(kPermBulkThreads, 2)
    permute_bulk_kernel(const T* __restrict__ in, long long in_rows,
                        const int* __restrict__ row_map, const int* __restrict__ col_map,
                        T* __restrict__ out, long long rows, int d, int* status) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) unsigned char bulk_smem[];
  constexpr int V = 16 / sizeof(T);
  constexpr int R = 8 / sizeof(T);
  constexpr int KR = 1;  // vectors whose table positions a thread keeps in registers
  const int nv = d / V;
  const int tid = threadIdx.x;
  const uint32_t row_bytes = static_cast<uint32_t>(d) * static_cast<uint32_t>(sizeof(T));
  const size_t tile = static_cast<size_t>(R) * row_bytes;  // one group: 8 d bytes
  uint2* ent = reinterpret_cast<uint2*>(bulk_smem + 2 * tile);
  uint64_t* full = reinterpret_cast<uint64_t*>(bulk_smem + 3 * tile);  // one per stage
  volatile int* abort_flag = reinterpret_cast<volatile int*>(full + 2);
  const long long groups = (rows + R - 1) / R;
  const long long count =
      blockIdx.x < groups ? (groups - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  // group n of this CTA: rows first_row(n) ..; stage n % 2, whose barrier
  // completes its (n / 2)-th phase when the group's rows have landed
  auto first_row = [&](long long n) { return (blockIdx.x + n * gridDim.x) * R; };
  auto stage = [&](long long n) { return bulk_smem + static_cast<size_t>(n & 1) * tile; };
  auto issue = [&](long long n) {  // thread 0: copy group n's source rows into its stage
    long long src[R];
    perm_group_sources<R>(first_row(n), rows, row_map, in_rows, src);
    uint32_t bytes = 0;
#pragma unroll
    for (int q = 0; q < R; ++q) bytes += src[q] >= 0 ? row_bytes : 0u;
    uint64_t* bar = &full[n & 1];
    mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
    for (int q = 0; q < R; ++q)
      if (src[q] >= 0) bulk_load_1d(stage(n) + q * row_bytes, in + src[q] * d, row_bytes, bar);
  };

  if (tid == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  long long issued = 0;  // thread 0: groups whose copies are issued
  if (tid == 0)
    for (; issued < 2 && issued < count; ++issued) issue(issued);

  uint32_t pos_r[KR][V / 2];
  bool bad_cols = false;
#pragma unroll
  for (int k = 0; k < KR; ++k) {
    const int v = tid + k * kPermBulkThreads;
#pragma unroll
    for (int i = 0; i < V / 2; ++i) pos_r[k][i] = 0xffffffffu;
    if (v < nv) bad_cols |= perm_table_positions<T>(col_map, v, d, nv, pos_r[k]);
  }
  if (bad_cols && count > 0) atomicCAS(status, 0, 1);

  long long n = 0;
  bool ok = true;
  for (; n < count; ++n) {
    unsigned char* st = stage(n);
    const long long r0 = first_row(n);
    long long src[R];
    if (perm_group_sources<R>(r0, rows, row_map, in_rows, src) && tid == 0)
      atomicCAS(status, 0, 1);
    const bool got = mbar_wait(&full[n & 1], static_cast<uint32_t>((n >> 1) & 1), abort_flag);
    if (!got) *abort_flag = 1;
    if (!__syncthreads_and(got)) {
      ok = false;
      break;
    }
    // interleave the staged rows into the table (rows without a source: 0)
    for (int v = tid; v < nv; v += kPermBulkThreads) {
      uint32_t wd[R][4];
#pragma unroll
      for (int q = 0; q < R; ++q) {
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (src[q] >= 0) w = *reinterpret_cast<const uint4*>(st + q * row_bytes + v * 16);
        wd[q][0] = w.x;
        wd[q][1] = w.y;
        wd[q][2] = w.z;
        wd[q][3] = w.w;
      }
      perm_store_entries<T>(ent, nv, v, wd);
    }
    // the stage has been read: the copies of group n + 2 go to it
    fence_proxy_async_shared();
    __syncthreads();
    if (tid == 0 && issued < count) {
      issue(issued);
      ++issued;
    }
    auto gather = [&](int v, const uint32_t (&pos)[V / 2]) {
      uint32_t o[R][4];
      perm_gather<T>(ent, pos, o);
#pragma unroll
      for (int q = 0; q < R; ++q)
        if (r0 + q < rows)
          reinterpret_cast<uint4*>(out + (r0 + q) * d)[v] =
              make_uint4(o[q][0], o[q][1], o[q][2], o[q][3]);
    };
#pragma unroll
    for (int k = 0; k < KR; ++k) {
      const int v = tid + k * kPermBulkThreads;
      if (v < nv) gather(v, pos_r[k]);
    }
    for (int v = tid + KR * kPermBulkThreads; v < nv; v += kPermBulkThreads) {
      uint32_t pos[V / 2];
      if (perm_table_positions<T>(col_map, v, d, nv, pos)) atomicCAS(status, 0, 1);
      gather(v, pos);
    }
    __syncthreads();  // the table is free
  }
  if (tid == 0) {
    if (!ok) {
      atomicCAS(status, 0, 5);  // POETX_ERR_TIMEOUT
      // let the copies still in flight land before the CTA exits
      for (long long m = n; m < issued; ++m) {
        const unsigned long long t0 = global_timer_ns();
        while (!mbar_try_wait(&full[m & 1], static_cast<uint32_t>((m >> 1) & 1)) &&
               global_timer_ns() - t0 < 10000000ull) {
        }
      }
    }
  }
}

// One Adam step on packed parameters: m, v moments, bias corrections bc1 =
// 1 - beta1^step and bc2 = 1 - beta2^step, decoupled weight decay wd.
__global__ void adam_kernel(float* __restrict__ theta, const float* __restrict__ grad,
                            float* __restrict__ m, float* __restrict__ v, long long n, float lr,
                            float beta1, float beta2, float eps, float wd, float bc1, float bc2) {
  pdl_wait();
  pdl_trigger();
  auto step1 = [&](float th, float g, float& mi, float& vi) {
    mi = beta1 * mi + (1.f - beta1) * g;
    vi = beta2 * vi + (1.f - beta2) * g * g;
    return th - lr * ((mi / bc1) / (sqrtf(vi / bc2) + eps) + wd * th);
  };
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long first = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  // 16-byte vectors where all four arrays allow them, the same arithmetic per element
  const bool vec = ((reinterpret_cast<uintptr_t>(theta) | reinterpret_cast<uintptr_t>(grad) |
                     reinterpret_cast<uintptr_t>(m) | reinterpret_cast<uintptr_t>(v)) & 15u) == 0;
  const long long n4 = vec ? n / 4 : 0;
  for (long long i = first; i < n4; i += stride) {
    const float4 g = reinterpret_cast<const float4*>(grad)[i];
    float4 mi = reinterpret_cast<float4*>(m)[i], vi = reinterpret_cast<float4*>(v)[i];
    float4 th = reinterpret_cast<float4*>(theta)[i];
    th.x = step1(th.x, g.x, mi.x, vi.x);
    th.y = step1(th.y, g.y, mi.y, vi.y);
    th.z = step1(th.z, g.z, mi.z, vi.z);
    th.w = step1(th.w, g.w, mi.w, vi.w);
    reinterpret_cast<float4*>(m)[i] = mi;
    reinterpret_cast<float4*>(v)[i] = vi;
    reinterpret_cast<float4*>(theta)[i] = th;
  }
  for (long long i = 4 * n4 + first; i < n; i += stride) {
    float mi = m[i], vi = v[i];
    theta[i] = step1(theta[i], grad[i], mi, vi);
    m[i] = mi;
    v[i] = vi;
  }
}

// ----------------------------------------------------- INT8 frozen weight
// One CTA of 256 threads per output row: absmax, scale = absmax / 127, then
// code = rint(w / scale) clamped to +-127 (float32 IEEE division; a zero row
// gets scale 0 and codes 0).
template <typename T>
__device__ __forceinline__ float load_f32(const T* p, long long i);
template <>
__device__ __forceinline__ float load_f32<float>(const float* p, long long i) {
  return p[i];
}
template <>
__device__ __forceinline__ float load_f32<__nv_bfloat16>(const __nv_bfloat16* p, long long i) {
  return __bfloat162float(p[i]);
}

template <typename T>
__global__ void __launch_bounds__(256) quantize_rows_kernel(const T* __restrict__ W,
                                                            int8_t* __restrict__ q,
                                                            float* __restrict__ scales, int d_in) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[8];
  const long long row0 = static_cast<long long>(blockIdx.x) * d_in;
  float amax = 0.f;
  for (int i = threadIdx.x; i < d_in; i += 256) amax = fmaxf(amax, fabsf(load_f32(W, row0 + i)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) amax = fmaxf(amax, red[w]);
  const float scale = amax > 0.f ? amax / 127.f : 0.f;
  if (threadIdx.x == 0) scales[blockIdx.x] = scale;
  for (int i = threadIdx.x; i < d_in; i += 256) {
    float c = scale > 0.f ? rintf(load_f32(W, row0 + i) / scale) : 0.f;
    c = fminf(fmaxf(c, -127.f), 127.f);
    q[row0 + i] = static_cast<int8_t>(static_cast<int>(c));
  }
}

// W[o][i] = code * scale[o] (one float32 product, rounded to T); sixteen
// codes per thread and 16-byte accesses when d_in % 16 == 0.
template <typename T>
__device__ __forceinline__ void store_16(T* dst, const float* v);
template <>
__device__ __forceinline__ void store_16<float>(float* dst, const float* v) {
  float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int j = 0; j < 4; ++j) d[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
}
template <>
__device__ __forceinline__ void store_16<__nv_bfloat16>(__nv_bfloat16* dst, const float* v) {
  uint32_t w[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
    w[j] = *reinterpret_cast<const uint32_t*>(&h);
  }
  uint4* d = reinterpret_cast<uint4*>(dst);
  d[0] = make_uint4(w[0], w[1], w[2], w[3]);
  d[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

template <typename T>
__global__ void dequantize_kernel(const int8_t* __restrict__ q, const float* __restrict__ scales,
                                  T* __restrict__ W, int d_in, long long total, int vec) {
  pdl_wait();
  pdl_trigger();
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  if (vec) {
    const long long chunks = total / 16;
    const unsigned per_row = static_cast<unsigned>(d_in / 16);  // d_in % 16 == 0: one row per chunk
    for (long long c = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; c < chunks;
         c += stride) {
      const long long e0 = c * 16;
      const long long row = chunks < (1ll << 32) ? static_cast<unsigned>(c) / per_row : c / per_row;
      const float s = scales[row];
      const int4 raw = reinterpret_cast<const int4*>(q)[c];
      const int words[4] = {raw.x, raw.y, raw.z, raw.w};
      float v[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int byte = (words[j >> 2] >> (8 * (j & 3))) & 0xff;
        v[j] = static_cast<float>(static_cast<int8_t>(byte)) * s;
      }
      store_16(W + e0, v);
    }
  } else {
    for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < total;
         e += stride)
      W[e] = from_f32<T>(static_cast<float>(q[e]) * scales[e / d_in]);
  }
}

int ew_grid(long long total) {
  long long blocks = (total + 255) / 256;
  const long long cap = static_cast<long long>(sm_count()) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return static_cast<int>(blocks);
}

}  // namespace

cudaError_t simt_gemm_run(const SimtGemm& g_in, cudaStream_t stream) {
  SimtGemm g = g_in;
  if (g.M <= 0 || g.N <= 0 || g.batches <= 0) return cudaSuccess;
  if (g.batches > 65535) return cudaErrorInvalidValue;
  const int tiles_n = (g.N + TN - 1) / TN, tiles_m = (g.M + TM - 1) / TM;
  if (tiles_m > 65535) return cudaErrorInvalidValue;
  // Small grids with long K: split K over a cluster of up to 8 CTAs per tile
  // (slices of at least one K step) until about two CTAs per SM work.
  const long long tiles = static_cast<long long>(tiles_n) * tiles_m * g.batches;
  int splits = 1;
  const long long want = 2LL * sm_count();
  while (splits < 8 && tiles * splits * 2 <= want && g.K >= 2 * splits * 32) splits *= 2;
  g.splits = splits;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(tiles_n * splits), static_cast<unsigned>(tiles_m),
                     static_cast<unsigned>(g.batches));
  cfg.blockDim = dim3(SIMT_THREADS);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(splits);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = splits > 1 ? 2 : 1;
  prof_begin(g.tag, stream);
  cudaError_t e = g.bf16_inputs ? cudaLaunchKernelEx(&cfg, simt_gemm_kernel<__nv_bfloat16>, g)
                                : cudaLaunchKernelEx(&cfg, simt_gemm_kernel<float>, g);
  prof_end(g.tag, stream);
  return e != cudaSuccess ? e : cudaGetLastError();
}

bool simt_fused_fits(int b) { return b >= 1 && b <= kFusedXW && (TK % b == 0 || b % TK == 0); }

cudaError_t simt_fused_run(const float* X, const float* L, bool l_trans, const float* W,
                           long long w_k, long long w_n, const float* R, bool r_trans, float* C,
                           float* out, int M, int N, int K, int b, const char* tag,
                           cudaStream_t stream) {
  if (M <= 0 || N <= 0 || K <= 0) return cudaSuccess;
  if (!simt_fused_fits(b) || N % b != 0 || K % b != 0 || (R != nullptr && out == nullptr))
    return cudaErrorInvalidValue;
  const int smem = kFusedSmemFloats * static_cast<int>(sizeof(float));
  void (*kernel)(const SimtFusedArgs) = nullptr;
  switch (b) {
    case 1: kernel = simt_fused_kernel<1>; break;
    case 2: kernel = simt_fused_kernel<2>; break;
    case 4: kernel = simt_fused_kernel<4>; break;
    case 8: kernel = simt_fused_kernel<8>; break;
    case 16: kernel = simt_fused_kernel<16>; break;
    case 32: kernel = simt_fused_kernel<32>; break;
    default: kernel = simt_fused_kernel<64>; break;
  }
  static bool attr_set[64] = {};
  static std::mutex mu;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64) {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_set[dev]) {  // every instance, once per device
      const void* all[] = {
          reinterpret_cast<const void*>(simt_fused_kernel<1>),
          reinterpret_cast<const void*>(simt_fused_kernel<2>),
          reinterpret_cast<const void*>(simt_fused_kernel<4>),
          reinterpret_cast<const void*>(simt_fused_kernel<8>),
          reinterpret_cast<const void*>(simt_fused_kernel<16>),
          reinterpret_cast<const void*>(simt_fused_kernel<32>),
          reinterpret_cast<const void*>(simt_fused_kernel<64>)};
      for (const void* f : all) {
        cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
      }
      attr_set[dev] = true;
    }
  }
  SimtFusedArgs a;
  a.M = M;
  a.N = N;
  a.K = K;
  a.b = b;
  a.X = X;
  a.L = L;
  a.l_trans = l_trans ? 1 : 0;
  a.W = W;
  a.w_k = w_k;
  a.w_n = w_n;
  a.R = R;
  a.r_trans = r_trans ? 1 : 0;
  a.C = C;
  a.out = out;
  const int tiles_n = (N + TN - 1) / TN, tiles_m = (M + TM - 1) / TM;
  if (tiles_m > 65535) return cudaErrorInvalidValue;
  // K split over a cluster of up to 8 CTAs per tile, as in simt_gemm_run
  const long long tiles = static_cast<long long>(tiles_n) * tiles_m;
  int splits = 1;
  while (splits < 8 && tiles * splits * 2 <= 2LL * sm_count() && K >= 2 * splits * 32)
    splits *= 2;
  a.splits = splits;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(tiles_n * splits), static_cast<unsigned>(tiles_m), 1);
  cfg.blockDim = dim3(SIMT_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(splits);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = splits > 1 ? 2 : 1;
  prof_begin(tag, stream);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, a);
  prof_end(tag, stream);
  return e != cudaSuccess ? e : cudaGetLastError();
}

#define POETX_EW_LAUNCH(tag, total, kernel, ...)                         \
  do {                                                                   \
    if ((total) <= 0) return cudaSuccess;                                \
    prof_begin(tag, s);                                                  \
    cudaError_t e_ = launch_pdl(kernel, dim3(ew_grid(total)), dim3(256), 0, s, __VA_ARGS__); \
    prof_end(tag, s);                                                    \
    return e_ != cudaSuccess ? e_ : cudaGetLastError();                  \
  } while (0)

cudaError_t launch_unpack(const float* theta_a, int n_a, const float* theta_b, int n_b, int b,
                          float* q32, __nv_bfloat16* q16, cudaStream_t s) {
  const int total = (n_a + n_b) * b * b;
  POETX_EW_LAUNCH("unpack", total, unpack_kernel, theta_a, n_a, theta_b, b, total, q32, q16);
}

cudaError_t launch_identity_plus(const float* q, int n, int b, float* o32, __nv_bfloat16* o16,
                                 cudaStream_t s) {
  const int total = n * b * b;
  POETX_EW_LAUNCH("identity_plus", total, identity_plus_kernel, q, b, total, o32, o16);
}

cudaError_t launch_expand_superblocks(const __nv_bfloat16* blocks, int n, int b, int S,
                                      __nv_bfloat16* out, cudaStream_t s) {
  const int per = S / b;
  const int nsb = (n + per - 1) / per;
  const int total8 = nsb * S * S / 8;  // 16-byte vectors
  if (b % 8 != 0 || S % b != 0 || reinterpret_cast<uintptr_t>(blocks) % 16 != 0 ||
      reinterpret_cast<uintptr_t>(out) % 16 != 0)
    return cudaErrorInvalidValue;
  POETX_EW_LAUNCH("expand_superblocks", total8, expand_superblocks_kernel, blocks, n, b, S, total8,
                  out);
}

cudaError_t launch_reduce_extract(const float* part, int splits, int n, int b, int S, float* o32,
                                  __nv_bfloat16* o16, cudaStream_t s) {
  const int total = n * b * b;
  POETX_EW_LAUNCH("reduce_extract", total, reduce_extract_kernel, part, splits, n, b, S, total,
                  o32, o16);
}

bool small_chain_fits(int b) { return b >= 1 && b <= kSmallMaxB; }

namespace {
cudaError_t small_outer_launch(const OuterSides& sides, int n, int b, long long T,
                               cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  if (!small_chain_fits(b) || n > 65535) return cudaErrorInvalidValue;
  // a cluster of up to 8 CTAs per block, a chunk of tokens at least each,
  // until about two CTAs per SM work
  int splits = 1;
  while (splits < 8 && static_cast<long long>(n) * splits * 2 <= 2LL * sm_count() &&
         T >= static_cast<long long>(splits) * 2 * kOuterTC)
    splits *= 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(splits), static_cast<unsigned>(n), 1);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(splits);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = splits > 1 ? 2 : 1;
  prof_begin("outer", s);
  cudaError_t e = cudaLaunchKernelEx(&cfg, small_outer_kernel, sides, b, T, splits);
  prof_end("outer", s);
  return e != cudaSuccess ? e : cudaGetLastError();
}
}  // namespace

cudaError_t launch_small_outer(const float* A, const float* B, float* G, int d, int b, long long T,
                               cudaStream_t s) {
  OuterSides sides = {{A, A}, {B, B}, {G, G}, {d, d}, 0};
  const int n = b > 0 ? d / b : 0;
  sides.n_a = n;
  return small_outer_launch(sides, n, b, T, s);
}

cudaError_t launch_small_outer2(const float* A0, const float* B0, float* G0, int d0,
                                const float* A1, const float* B1, float* G1, int d1, int b,
                                long long T, cudaStream_t s) {
  if (b <= 0) return cudaErrorInvalidValue;
  OuterSides sides = {{A0, A1}, {B0, B1}, {G0, G1}, {d0, d1}, d0 / b};
  return small_outer_launch(sides, d0 / b + d1 / b, b, T, s);
}

cudaError_t launch_small_build(const float* theta, int n, int b, int k, float* out32,
                               __nv_bfloat16* out16, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  if (!small_chain_fits(b)) return cudaErrorInvalidValue;
  const size_t smem = 3ull * b * b * sizeof(float);  // at most 48 KiB
  prof_begin("build", s);
  cudaError_t e = launch_pdl(small_build_kernel, dim3(static_cast<unsigned>(n)), dim3(256), smem, s,
                             theta, b, k, out32, out16);
  prof_end("build", s);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_small_adjoint(const float* theta_a, int n_a, const float* theta_b, int n_b,
                                 int b, int k, const float* G, float* dtheta_a, float* dtheta_b,
                                 cudaStream_t s) {
  if (n_a + n_b <= 0) return cudaSuccess;
  if (!small_chain_fits(b)) return cudaErrorInvalidValue;
  const size_t smem = 6ull * b * b * sizeof(float);  // at most 96 KiB
  static bool attr_set[64] = {};
  static std::mutex mu;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64) {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_set[dev]) {
      cudaFuncSetAttribute(small_adjoint_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           6 * kSmallMaxB * kSmallMaxB * static_cast<int>(sizeof(float)));
      attr_set[dev] = true;
    }
  }
  prof_begin("cnp_bwd", s);
  cudaError_t e = launch_pdl(small_adjoint_kernel, dim3(static_cast<unsigned>(n_a + n_b)),
                             dim3(256), smem, s, theta_a, n_a, theta_b, b, k, G, dtheta_a,
                             dtheta_b);
  prof_end("cnp_bwd", s);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_pack_skew(const float* A, const float* B, int n_a, int n_b, int b,
                             float* dtheta_a, float* dtheta_b, cudaStream_t s) {
  const int total = (n_a + n_b) * b * b;
  POETX_EW_LAUNCH("pack_skew", total, pack_skew_kernel, A, B, n_a, b, total, dtheta_a, dtheta_b);
}

cudaError_t launch_prep_tiles(const PrepTilesArgs& a, cudaStream_t s) {
  if (a.b % TT != 0 || a.n_a + a.n_b <= 0) return cudaErrorInvalidValue;
  const int t = a.b / TT;
  dim3 grid(t * (t + 1) / 2, a.n_a + a.n_b);
  prof_begin("prep_tiles", s);
  cudaError_t e = launch_pdl(prep_tiles_kernel, grid, dim3(256), 0, s, a);
  prof_end("prep_tiles", s);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_pack_tiles(const float* D, float sign, int n_a, int n_b, int b,
                              float* dtheta_a, float* dtheta_b, cudaStream_t s) {
  if (b % TT != 0 || n_a + n_b <= 0) return cudaErrorInvalidValue;
  const int t = b / TT;
  dim3 grid(t * (t + 1) / 2, n_a + n_b);
  prof_begin("pack_tiles", s);
  cudaError_t e = launch_pdl(pack_tiles_kernel, grid, dim3(256), 0, s, D, sign, n_a, b,
                             dtheta_a, dtheta_b);
  prof_end("pack_tiles", s);
  return e != cudaSuccess ? e : cudaGetLastError();
}

namespace {
// One launch of an index-map kernel with as many CTAs as fit at once (the
// maximum shared-memory carveout, set once per device and kernel: one
// instance of this function per kernel).
template <typename T, auto kernel>
cudaError_t permute_launch(int threads, size_t smem, const void* in, long long in_rows,
                           const int* row_map, const int* col_map, void* out, long long rows,
                           int d, cudaStream_t s) {
  constexpr int R = 8 / sizeof(T);
  const long long groups = (rows + R - 1) / R;
  const void* fn = reinterpret_cast<const void*>(kernel);
  static bool attr_set[64] = {};
  static std::mutex mu;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64) {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_set[dev]) {
      cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kPermSmemMax));
      attr_set[dev] = true;
    }
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const long long cap = static_cast<long long>(sm_count()) * per_sm;
  const dim3 grid(static_cast<unsigned>(groups < cap ? groups : cap));
  return launch_pdl(kernel, grid, dim3(threads), smem, s, static_cast<const T*>(in), in_rows,
                    row_map, col_map, static_cast<T*>(out), rows, d, device_status_ptr());
}

template <typename T>
cudaError_t permute_dispatch(const void* in, long long in_rows, const int* row_map,
                             const int* col_map, void* out, long long rows, int d,
                             cudaStream_t s) {
  const size_t table = static_cast<size_t>(d) * 8;  // one 8-byte entry per column
  if (perm_bulk_smem(d) <= kPermSmemMax)
    return permute_launch<T, permute_bulk_kernel<T>>(kPermBulkThreads, perm_bulk_smem(d), in,
                                                      in_rows, row_map, col_map, out, rows, d, s);
  if (2 * table <= kPermSmemMax)  // two tables: loads overlap the gather
    return permute_launch<T, permute_rows_kernel<T, 2>>(kPermThreads, 2 * table, in, in_rows,
                                                         row_map, col_map, out, rows, d, s);
  return permute_launch<T, permute_rows_kernel<T, 1>>(kPermThreads, table, in, in_rows, row_map,
                                                       col_map, out, rows, d, s);
}
}  // namespace

cudaError_t launch_permute_rows(const void* in, long long in_rows, const int* row_map,
                                const int* col_map, void* out, long long rows, int d,
                                bool is_bf16, cudaStream_t s) {
  if (rows <= 0 || d <= 0) return cudaSuccess;
  if (static_cast<size_t>(d) * 8 > kPermSmemMax) return cudaErrorInvalidValue;
  prof_begin("permute", s);
  const cudaError_t e =
      is_bf16 ? permute_dispatch<__nv_bfloat16>(in, in_rows, row_map, col_map, out, rows, d, s)
              : permute_dispatch<float>(in, in_rows, row_map, col_map, out, rows, d, s);
  prof_end("permute", s);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_adam(float* theta, const float* grad, float* m, float* v, long long n,
                        float lr, float beta1, float beta2, float eps, float wd, float bc1,
                        float bc2, cudaStream_t s) {
  // one thread per 16-byte vector (a grid-stride loop covers the rest)
  POETX_EW_LAUNCH("adam", (n + 3) / 4, adam_kernel, theta, grad, m, v, n, lr, beta1, beta2, eps, wd, bc1,
                  bc2);
}

cudaError_t launch_quantize_rows(const void* W, bool is_bf16, int8_t* q, float* scales, int d_in,
                                 int d_out, cudaStream_t s) {
  if (d_in <= 0 || d_out <= 0) return cudaSuccess;
  prof_begin("quantize", s);
  cudaError_t e =
      is_bf16 ? launch_pdl(quantize_rows_kernel<__nv_bfloat16>, dim3(d_out), dim3(256), 0, s,
                           static_cast<const __nv_bfloat16*>(W), q, scales, d_in)
              : launch_pdl(quantize_rows_kernel<float>, dim3(d_out), dim3(256), 0, s,
                           static_cast<const float*>(W), q, scales, d_in);
  prof_end("quantize", s);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_dequantize(const int8_t* q, const float* scales, void* W, bool is_bf16,
                              int d_in, int d_out, cudaStream_t s) {
  const long long total = static_cast<long long>(d_in) * d_out;
  if (total <= 0) return cudaSuccess;
  const int vec = (d_in % 16 == 0 && reinterpret_cast<uintptr_t>(q) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(W) % 16 == 0)
                      ? 1
                      : 0;
  const long long items = vec ? total / 16 : total;
  long long blocks = (items + 255) / 256;
  // enough threads for one 16-code chunk each at 4096 x 4096 (all loads in flight at once)
  const long long cap = static_cast<long long>(sm_count()) * 32;
  if (blocks > cap) blocks = cap;
  prof_begin("dequantize", s);
  cudaError_t e =
      is_bf16 ? launch_pdl(dequantize_kernel<__nv_bfloat16>, dim3(static_cast<unsigned>(blocks)),
                           dim3(256), 0, s, q, scales, static_cast<__nv_bfloat16*>(W), d_in,
                           total, vec)
              : launch_pdl(dequantize_kernel<float>, dim3(static_cast<unsigned>(blocks)),
                           dim3(256), 0, s, q, scales, static_cast<float*>(W), d_in, total, vec);
  prof_end("dequantize", s);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_f32_to_bf16(const float* in, long long count, __nv_bfloat16* out,
                               cudaStream_t s) {
  POETX_EW_LAUNCH("f32_to_bf16", count, f32_to_bf16_kernel, in, count, out);
}

}  // namespace poetx
