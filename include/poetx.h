/*
 * poetx.h -- C ABI of the POET-X layer hot path on one NVIDIA GB300 (sm_103a).
 *
 * POET-X trains each weight as W = R * W0 * P with W0 frozen and R, P
 * orthogonal, so the singular values of W0 are preserved (arXiv 2603.05500
 * abstract, "POET-X: Memory-efficient LLM Training by Scaling Orthogonal
 * Transformation"; gist.science technical summary of that paper, section 1,
 * "Vorarbeit (POET)").  R and P are block diagonal with b x b blocks; each
 * block is the Cayley transform of a skew-symmetric Q with the inverse
 * replaced by a Neumann series cut after Q^k, and only the strict upper
 * triangle of Q is stored (same summary, section 2, "Effiziente
 * Cayley-Neumann-Parametrisierung (CNP)" and "Batch-parallele Berechnung
 * fuer Block-diagonale Matrizen").  The transforms are applied to the
 * activations, never to W0 (section 2, "Input-zentrische Implementierung"):
 *
 *     y_t = R (W0 (P x_t))          for every token t
 *
 * Conventions shared by every entry point
 *   - Activations are token-major, row-major: x[t][i] at x + t*d_in + i.
 *   - W0 is [d_out][d_in] row-major (v_t = W0 u_t).
 *   - Packed parameters theta: [d/b][b(b-1)/2] float32; block g's entry
 *     (i, j), i < j, sits at g*b(b-1)/2 + i*b - i(i+1)/2 + (j-i-1), and
 *     Q[j][i] = -Q[i][j], Q[i][i] = 0.
 *   - Blocks: [d/b][b][b] row-major in the working dtype; block g maps
 *     features g*b .. g*b+b-1: z[g*b+i] = sum_j B_g[i][j] x[g*b+j].
 *   - dtype POETX_BF16: activations, W0 and blocks are bfloat16, every
 *     contraction accumulates in fp32 on the tensor cores (tcgen05).
 *     POETX_F32: everything float32, fp32 FFMA on the CUDA cores.
 *   - All pointers are device pointers, 16-byte aligned, owned by the
 *     caller.  The library allocates no device memory and keeps no state
 *     besides a per-device status word; scratch comes from the caller's
 *     workspace, whose size the *_workspace_size functions return.
 *   - Every call only enqueues work on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream) and returns; results are ready when the stream
 *     is.  Calls on one stream may share one workspace; calls that may run
 *     concurrently need separate workspaces.
 *   - Supported shapes: b >= 2, b <= 512, d % b == 0 for F32.  BF16 also
 *     needs b in {32, 64, 128, 256, 512} and every feature dimension a
 *     multiple of max(b, 256) (POETX_ERR_UNSUPPORTED otherwise).  0 <= k
 *     <= 16.  0 <= tokens <= 2^22; with tokens = 0 the activation pointers
 *     may be NULL and outputs that are sums over tokens are set to zero.
 *   - Errors: argument problems return POETX_ERR_INVALID_ARG /
 *     UNSUPPORTED / WORKSPACE before anything is enqueued; a launch failure
 *     returns POETX_ERR_CUDA.  A kernel that gives up on an internal wait
 *     records POETX_ERR_TIMEOUT in the status word, read with
 *     poetx_device_status().
 */
#ifndef POETX_H_
#define POETX_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  POETX_OK = 0,
  POETX_ERR_INVALID_ARG = 1,
  POETX_ERR_UNSUPPORTED = 2,
  POETX_ERR_WORKSPACE = 3,
  POETX_ERR_CUDA = 4,
  POETX_ERR_TIMEOUT = 5
} poetx_status;

typedef enum { POETX_F32 = 0, POETX_BF16 = 1 } poetx_dtype;

typedef void* poetx_stream; /* cudaStream_t */

/* Human-readable name of a status code (static storage). */
const char* poetx_status_string(poetx_status s);

/* Number of float32 parameters of one side: (d/b) * b(b-1)/2 ("only the
 * upper triangle of the skew-symmetric Q is stored", technical summary,
 * section 2, CNP bullet).  Returns 0 for invalid d, b. */
size_t poetx_packed_size(int d, int b);

/* ------------------------------------------------------------------------
 * Block build: packed theta -> blocks R_k(Q_g) = (I + Q)(I + Q + ... + Q^k)
 *   = I + 2Q + ... + 2Q^k + Q^{k+1}, the Neumann-truncated Cayley transform
 * (technical summary, section 2, CNP bullet: the powers Q^2..Q^4 of k = 3
 * are built in one fused step).  Arithmetic in fp32 (F32) or bf16 tensor
 * cores with fp32 accumulation (BF16: b >= 128, and 1 <= k <= 16 with
 * b = 32..256);
 * rounded once at the store.
 *   theta  [d/b][b(b-1)/2] float32 (read only)
 *   blocks [d/b][b][b] dtype (written)
 * Blocks are independent, so both factors of a layer are one call when
 * theta_P and theta_R lie back to back (and the blocks likewise):
 * d = d_in + d_out builds P's blocks then R's, bitwise as two calls would.
 * BF16 with 1 <= k <= 16 and b <= 256 runs on CTA pairs with every
 * operand in shared memory and needs no workspace (its size is 0 and the
 * workspace may be NULL).
 * ------------------------------------------------------------------------ */
size_t poetx_build_workspace_size(int d, int b, int k, poetx_dtype dtype);
poetx_status poetx_build_blocks(const float* theta, int d, int b, int k, poetx_dtype dtype,
                                void* blocks, void* workspace, size_t workspace_bytes,
                                poetx_stream stream);

/* Block build for callers that cannot allocate device memory.  The paper has
 * no counterpart: this is a convenience of this library.  Callers running
 * under a memory plan that forbids new allocations, or that own every
 * device buffer and have no workspace to offer, can build blocks here
 * without passing a workspace.  Same arithmetic and kernels as
 * poetx_build_blocks; the scratch is one fixed device array of the library
 * (12 MiB + 1 KiB, held on every GPU that loads the library until the
 * process exits), so:
 *   - (d/b) * b * b = d * b must be <= 2^20 (e.g. d = 4096 with b = 256);
 *     larger builds return POETX_ERR_WORKSPACE before anything is enqueued;
 *   - each call made outside stream capture looks up that array's device
 *     address (cudaGetSymbolAddress) with the device current, so the
 *     address stays right after the context is re-created (for example by
 *     cudaDeviceReset); a call made while its stream is being captured
 *     reuses the address of the last call outside capture on that device,
 *     so make the first call on a device, and the first after a device
 *     reset, before any stream capture (otherwise POETX_ERR_CUDA);
 *   - calls share the array: calls that overlap on the GPU (other streams
 *     or host threads on the same device) race and must be serialised;
 *     nothing needs to be zeroed between calls.
 * Allocates no device memory. */
poetx_status poetx_build_blocks_noalloc(const float* theta, int d, int b, int k, poetx_dtype dtype,
                                        void* blocks, poetx_stream stream);

/* ------------------------------------------------------------------------
 * Forward: y_t = R (W0 (P x_t)) (technical summary, section 2,
 * "Input-zentrische Implementierung" and the block-diagonal bullet).
 *   x       [tokens][d_in]   dtype (read)
 *   W0      [d_out][d_in]    dtype (read; frozen)
 *   P_blocks [d_in/b][b][b], R_blocks [d_out/b][b][b]  dtype (read)
 *   y       [tokens][d_out]  dtype (written)
 *   v_saved [tokens][d_out]  dtype, v_t = W0 P x_t, written if not NULL
 *           (the backward pass needs it; pass NULL to have it recomputed)
 * ------------------------------------------------------------------------ */
size_t poetx_forward_workspace_size(int d_in, int d_out, int b, int64_t tokens,
                                    poetx_dtype dtype);
poetx_status poetx_forward(const void* x, const void* W0, const void* P_blocks,
                           const void* R_blocks, void* y, void* v_saved, int d_in, int d_out,
                           int b, int64_t tokens, poetx_dtype dtype, void* workspace,
                           size_t workspace_bytes, poetx_stream stream);

/* ------------------------------------------------------------------------
 * Backward of L = sum_t <dy_t, y_t> with W0 frozen:
 *   dx_t = P^T W0^T R^T dy_t,
 *   dtheta_P, dtheta_R = d L / d theta for the packed parameters, i.e. the
 *   adjoint of the Cayley-Neumann polynomial applied to the block gradient
 *   G = sum_t (dout_t)(in_t)^T, then skew-projected and packed:
 *   dtheta[idx(i,j)] = G_Q[i][j] - G_Q[j][i].
 *   dy [tokens][d_out], x [tokens][d_in], W0, blocks: dtype (read)
 *   theta_P, theta_R: packed float32 (read)
 *   v_saved [tokens][d_out] from poetx_forward, or NULL: v is recomputed
 *           from x (activation recompute, the POET-Xmem trade of memory for
 *           time: technical summary, section 2, "Gradient Checkpointing")
 *   dx [tokens][d_in] dtype, dtheta_P, dtheta_R float32: overwritten
 * ------------------------------------------------------------------------ */
size_t poetx_backward_workspace_size(int d_in, int d_out, int b, int k, int64_t tokens,
                                     poetx_dtype dtype, int recompute_v);
poetx_status poetx_backward(const void* dy, const void* x, const void* W0, const float* theta_P,
                            const float* theta_R, const void* P_blocks, const void* R_blocks,
                            const void* v_saved, void* dx, float* dtheta_P, float* dtheta_R,
                            int d_in, int d_out, int b, int k, int64_t tokens, poetx_dtype dtype,
                            void* workspace, size_t workspace_bytes, poetx_stream stream);

/* ------------------------------------------------------------------------
 * Isolated block-diagonal transform z_t = B x_t and its backward (the
 * block-parallel product of the technical summary, section 2, on its own):
 *   forward : out [tokens][d] = blockdiag(blocks) applied to x [tokens][d]
 *   backward: dx_t = B^T dout_t and dtheta = packed d L / d theta for
 *             L = sum_t <dout_t, z_t>
 * ------------------------------------------------------------------------ */
size_t poetx_transform_workspace_size(int d, int b, int k, int64_t tokens, poetx_dtype dtype);
poetx_status poetx_transform_forward(const void* x, const void* blocks, void* out, int d, int b,
                                     int64_t tokens, poetx_dtype dtype, void* workspace,
                                     size_t workspace_bytes, poetx_stream stream);
poetx_status poetx_transform_backward(const void* dout, const void* x, const float* theta,
                                      const void* blocks, void* dx, float* dtheta, int d, int b,
                                      int k, int64_t tokens, poetx_dtype dtype, void* workspace,
                                      size_t workspace_bytes, poetx_stream stream);

/* ------------------------------------------------------------------------
 * Permuted blocks (technical summary, section 2, "Permutations-Beschleunigung
 * und -Reduktion"): POET mixes the blocks as R = Pi_R^T B_R Pi_R and
 * P = Pi_P^T B_P Pi_P; POET-X applies the permutations to the data as index
 * maps and folds the two inner ones into the weight once, so that
 *     y = Pi_R^T B_R W0' B_P Pi_P x,   W0' = Pi_R W0 Pi_P^T.
 * A permuted step is: x' = Pi_P x, the plain forward/backward on
 * (x', W0', blocks), y = Pi_R^T y', dy' = Pi_R dy, dx = Pi_P^T dx'; the
 * packed gradients come out of the plain backward unchanged.
 *   perm arrays: int32 device arrays holding a permutation of 0..d-1
 *   (16-byte aligned like every other pointer; perm_out of the fold needs
 *   only 4); (Pi x)[i] = x[perm[i]], so Pi^T is applied with the inverse
 *   permutation.
 *   Entries outside 0..d-1 are not followed: the output gets 0 and
 *   POETX_ERR_INVALID_ARG is recorded in the status word.  Rows must be a
 *   multiple of 16 bytes and d <= 28672 (INVALID_ARG otherwise).
 * ------------------------------------------------------------------------ */
/* out[r][i] = in[r][perm[i]] for rows x d activations (in != out). */
poetx_status poetx_permute_features(const void* in, const int32_t* perm, void* out, int64_t rows,
                                    int d, poetx_dtype dtype, poetx_stream stream);
/* W0_folded[i][j] = W0[perm_out[i]][perm_in[j]], i.e. Pi_R W0 Pi_P^T with
 * perm_out = the permutation of R and perm_in = the permutation of P. */
poetx_status poetx_fold_permutations(const void* W0, const int32_t* perm_out,
                                     const int32_t* perm_in, void* W0_folded, int d_in,
                                     int d_out, poetx_dtype dtype, poetx_stream stream);

/* ------------------------------------------------------------------------
 * Around the layer step.
 * Merge (technical summary, section 2, "Input-zentrische Implementierung":
 * the original POET updates the weight itself, W <- R W P): folds the
 * current blocks into the frozen weight, W0_out = R W0 P, and restarts the
 * factors from the identity by zeroing theta_P / theta_R when they are not
 * NULL (rebuild the blocks afterwards).  W0_out may be W0.
 *   W0, W0_out [d_out][d_in] dtype; blocks as for poetx_forward.
 * ------------------------------------------------------------------------ */
size_t poetx_merge_workspace_size(int d_in, int d_out, int b, poetx_dtype dtype);
poetx_status poetx_merge(const void* W0, const void* P_blocks, const void* R_blocks, void* W0_out,
                         float* theta_P, float* theta_R, int d_in, int d_out, int b,
                         poetx_dtype dtype, void* workspace, size_t workspace_bytes,
                         poetx_stream stream);
/* One Adam step (bias-corrected, decoupled weight decay) on n packed
 * parameters, in place: m <- b1 m + (1-b1) g; v <- b2 v + (1-b2) g^2;
 * theta <- theta - lr (m/(1-b1^step) / (sqrt(v/(1-b2^step)) + eps) + wd theta).
 * The pages name no optimizer for theta; this is the plain choice.  All
 * arrays float32 device memory; step >= 1. */
poetx_status poetx_adam_update(float* theta, const float* grad, float* m, float* v, int64_t n,
                               int step, float lr, float beta1, float beta2, float eps,
                               float weight_decay, poetx_stream stream);

/* ------------------------------------------------------------------------
 * INT8 frozen weight (POET-XQ; technical summary, section 2, "Quantisierte
 * Unterstuetzung (POET-XQ)": W0 is only the operand of one matmul, so it can
 * be held quantised).  Symmetric, one scale per output row:
 *   scale[o] = max_i |W0[o][i]| / 127   (float32; 0 for a zero row)
 *   W0_q[o][i] = rint(W0[o][i] / scale[o]) clamped to [-127, 127]
 *   (float32 IEEE division, ties to even).
 * Dequantisation writes W0[o][i] = W0_q[o][i] * scale[o] (one float32
 * product, rounded to dtype), the operand the forward and backward take.
 *   W0, W0_q [d_out][d_in] row-major; scales [d_out] float32.
 * d_in == 0 or d_out == 0 is a no-op; NULL pointers are INVALID_ARG.
 * ------------------------------------------------------------------------ */
poetx_status poetx_quantize_w0(const void* W0, int8_t* W0_q, float* scales, int d_in, int d_out,
                               poetx_dtype dtype, poetx_stream stream);
poetx_status poetx_dequantize_w0(const int8_t* W0_q, const float* scales, void* W0, int d_in,
                                 int d_out, poetx_dtype dtype, poetx_stream stream);

/* The W0 GEMM fused with the block-diagonal factors (technical summary,
 * section 2, input-centric bullet; the fusion itself is this library's):
 * with fusion on, poetx_forward computes y = R v in the epilogue of the
 * GEMM that produces v (v is stored only into a non-NULL v_saved), and
 * poetx_backward computes dx = du P in the epilogue of the GEMM that
 * produces du, for BF16 with b <= 256; the token sums of the P side then
 * run on their own over x and du.  y and everything on the R side have the
 * same bits as the unfused path; dx and dtheta_P agree to fp32 summation
 * order.  Off by default: on GB300 the fused W0 GEMM on CTA pairs takes
 * about 55 us longer per launch at d = 4096, T = 16384 (the block product
 * adds 6 % of MMA work, and staging the tile twice in TMEM reads, shared
 * memory and TMA stores slows the main loop), more than the separate block
 * transform it replaces.  Process-wide; returns the previous setting. */
int poetx_set_block_epilogue_fusion(int enable);

/* Scheduling of the W0 GEMMs (technical summary, section 2: the frozen-
 * weight product; the schedule is this library's).  The GEMMs run as
 * clusters of two CTAs, each cluster on two 128 x 256 output tiles at a
 * time.  When the last round keeps at most half of the clusters busy (r
 * pairs of tiles with 2r <= clusters) and K is an even number of 64-wide
 * steps, its 2r tiles are spread one per cluster and each cluster's two CTAs
 * sum the two halves of K, which the epilogue adds: the round takes half as
 * long.  GEMMs with at most half as many tile pairs as clusters run split
 * entirely.  That changes the fp32 summation order of those tiles only,
 * so v and du agree with the unsplit schedule to rounding; with the split
 * off every tile sums K in order in one CTA and the results do not depend
 * on the GPU's SM count.  On by default.  Process-wide; returns the
 * previous setting. */
int poetx_set_w0_split_tail(int enable);

/* The MMA form of the W0 GEMMs (technical summary, section 2: the frozen-
 * weight product; the kernel form is this library's).  On: each cluster of
 * two CTAs computes 256 x 256 output tiles with one tcgen05 MMA per 16-wide
 * K slice spanning both SMs (each SM holds 128 rows of the input tile and
 * half of the W0 tile, so it loads 32 KiB per 64-wide K step instead of
 * 48 KiB); the split of the last round (poetx_set_w0_split_tail) does not
 * apply.  Off: the clusters of two one-SM MMAs described above.  Both sum
 * K in order per output element; results agree to fp32 summation order.
 * On by default.  Process-wide; returns the previous setting. */
int poetx_set_w0_pair_mma(int enable);

/* ------------------------------------------------------------------------
 * Status and measurement
 * ------------------------------------------------------------------------ */
/* Synchronizes the current device, returns the status recorded by kernels
 * since the last call (POETX_OK or POETX_ERR_TIMEOUT) and clears it;
 * POETX_ERR_CUDA if the device reports an error. */
poetx_status poetx_device_status(void);

/* Self-check of the timeout path: enqueues one kernel whose barrier wait is
 * never satisfied; after limit_us microseconds (1..10^6) the wait gives up,
 * records POETX_ERR_TIMEOUT in the status word and the kernel returns.  A
 * following poetx_device_status() reports POETX_ERR_TIMEOUT once and the
 * context stays usable.  (No counterpart on the pages: library plumbing.) */
poetx_status poetx_selftest_wait_timeout(unsigned int limit_us, poetx_stream stream);

/* Total number of kernels this library has launched in this process. */
long long poetx_launch_count(void);

/* Launch timing: while on, every launch is bracketed by CUDA events on its
 * own stream, grouped by kernel tag ("gemm_w0", "transform", ...).
 * poetx_profile_start(capacity) clears earlier records and turns timing on
 * for up to `capacity` launches; poetx_profile_stop() turns it off.
 * poetx_profile_query(tag, &count, &total_ms) synchronizes the recorded
 * events and sums the durations of launches with that tag (NULL = all).
 * Returns 0, or -1 if no events could be created. */
int poetx_profile_start(int capacity);
void poetx_profile_stop(void);
int poetx_profile_query(const char* tag, int* count, double* total_ms);

#ifdef __cplusplus
}
#endif

#endif /* POETX_H_ */
