"""Float64 CPU oracle for the POET-X layer: packed skew generators, the
Cayley-Neumann block build, y = R_b (W0 (P_b x)) and its backward.

TEST INFRASTRUCTURE ONLY.  This module exists to check the CUDA library.
Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import it; the library itself never calls it and has no CPU fallback.  It
shares no code with the CUDA sources.

Everything is plain numpy in float64; ``@`` (a library matmul) and
``numpy.linalg.solve`` are the only library steps.  Nothing is blocked,
fused or reordered beyond the formulas below.

Sources (one web page each; the method's own paper is not available):
  [abstract]  arXiv 2603.05500 abstract, "POET-X: Memory-efficient LLM
              Training by Scaling Orthogonal Transformation": POET optimises
              each weight by an orthogonal equivalence transformation that
              preserves its spectrum.
  [tech-1]    gist.science summary of the same paper, "Technische
              Zusammenfassung", section 1 (Problemstellung, "Vorarbeit
              (POET)"): W = R W0 P with trainable orthogonal R and P.
  [tech-2-in] same page, section 2 (Methodik), bullet "Input-zentrische
              Implementierung": apply the transforms to activations, never
              form the merged weight.
  [tech-2-bd] section 2, bullet "Batch-parallele Berechnung fuer
              Block-diagonale Matrizen": R and P are block diagonal; the
              blocks are independent matrices multiplied as a batch.
  [tech-2-merge] section 2, bullet "Input-zentrische Implementierung": the
              original POET updates the weight itself, W <- R W P; here the
              same merge folds the trained factors into W0 (and the factors
              restart from the identity, theta = 0).
  [tech-2-perm] section 2, bullet "Permutations-Beschleunigung und
              -Reduktion": POET mixes the blocks with permutation matrices;
              POET-X applies the permutations as index maps on the data and
              folds two of the four forward permutations into W once.
  [tech-2-xq] section 2, bullet "Quantisierte Unterstuetzung (POET-XQ)":
              the frozen W0 is needed only as the operand of one matmul, so
              it can be held quantised (INT8) without more activation memory.
  [tech-2-cnp] section 2, bullet "Effiziente Cayley-Neumann-
              Parametrisierung (CNP)": the orthogonal blocks come from
              skew-symmetric Q (Q = -Q^T) through the Cayley transform with
              a Neumann-series inverse; only the upper triangle of Q is
              stored; the powers Q^2, Q^3, Q^4 are the work of one fused
              kernel.

Readings taken where the pages are silent (each one is listed with its
reason in the design notes):
  * Cayley form C(Q) = (I+Q)(I-Q)^{-1}; the Neumann truncation after Q^k
    replaces (I-Q)^{-1} by I+Q+...+Q^k, so a block is
    R_k(Q) = (I+Q)(I+Q+...+Q^k) = I + 2Q + ... + 2Q^k + Q^{k+1}.
    k = 3 gives the Q^2, Q^3, Q^4 of [tech-2-cnp].
  * The packed vector holds the strict upper triangle row by row
    (i < j; row i, then j ascending), Q[j][i] = -Q[i][j], zero diagonal.
  * Activations are token-major [T][d]; W0 is [d_out][d_in]; per token
    y_t = R (W0 (P x_t)).
  * The gradient returned for the packed parameters is d loss / d theta:
    dtheta[idx(i,j)] = G_Q[i][j] - G_Q[j][i].
  * INT8 W0 [tech-2-xq]: symmetric, one scale per output row,
    scale = max|W0[o,:]| / 127, code = round-half-even(W0 / scale) clamped
    to [-127, 127]; a row whose scale is 0 has codes 0.  The quotient that
    decides each code, and the dequantised value code * scale, are taken in
    float32 (the precision of the kernels), so codes are exact to compare.
"""

from __future__ import annotations

import numpy as np


# --------------------------------------------------------------------------
# Packed upper triangle  [tech-2-cnp]
# --------------------------------------------------------------------------

def packed_size(b: int) -> int:
    """Number of free parameters of a b x b skew-symmetric block."""
    return b * (b - 1) // 2


def packed_index(i, j, b: int):
    """Position of Q[i][j] (0 <= i < j < b) in the row-by-row strict upper
    triangle: rows 0..i-1 hold (b-1) + (b-2) + ... + (b-i) entries."""
    i = np.asarray(i)
    j = np.asarray(j)
    return i * b - (i * (i + 1)) // 2 + (j - i - 1)


def unpack(theta: np.ndarray, b: int) -> np.ndarray:
    """theta [n][b(b-1)/2] -> skew-symmetric Q [n][b][b] (float64)."""
    theta = np.asarray(theta, dtype=np.float64)
    n = theta.shape[0]
    assert theta.shape == (n, packed_size(b))
    ii, jj = np.triu_indices(b, 1)
    idx = packed_index(ii, jj, b)
    Q = np.zeros((n, b, b), dtype=np.float64)
    Q[:, ii, jj] = theta[:, idx]
    Q[:, jj, ii] = -theta[:, idx]
    return Q


def pack_skew_grad(G_Q: np.ndarray) -> np.ndarray:
    """Gradient of a loss with respect to the packed parameters, given its
    gradient G_Q with respect to an unconstrained Q: theta feeds Q[i][j]
    with +1 and Q[j][i] with -1."""
    n, b, _ = G_Q.shape
    ii, jj = np.triu_indices(b, 1)
    out = np.zeros((n, packed_size(b)), dtype=np.float64)
    out[:, packed_index(ii, jj, b)] = G_Q[:, ii, jj] - G_Q[:, jj, ii]
    return out


# --------------------------------------------------------------------------
# Cayley-Neumann blocks  [tech-2-cnp]
# --------------------------------------------------------------------------

def neumann_coefficients(k: int) -> np.ndarray:
    """c_i of R_k(Q) = sum_i c_i Q^i, i = 0..k+1:  (I+Q) * sum_{i<=k} Q^i."""
    c = np.zeros(k + 2)
    c[: k + 1] += 1.0      # I + Q + ... + Q^k
    c[1: k + 2] += 1.0     # Q * (I + Q + ... + Q^k)
    return c


def matrix_powers(Q: np.ndarray, m: int) -> list:
    """[Q^0, Q^1, ..., Q^m] for a stack of square matrices."""
    n, b, _ = Q.shape
    P = [np.broadcast_to(np.eye(b), (n, b, b)).copy()]
    for _ in range(m):
        P.append(P[-1] @ Q)
    return P


def cayley_neumann(Q: np.ndarray, k: int) -> np.ndarray:
    """R_k = (I + Q)(I + Q + ... + Q^k), explicit powers."""
    pw = matrix_powers(Q, k)
    S = sum(pw)
    return (pw[0] + Q) @ S


def cayley_exact(Q: np.ndarray) -> np.ndarray:
    """C = (I+Q)(I-Q)^{-1} = (I-Q)^{-1}(I+Q): solve (I-Q) C = I+Q."""
    n, b, _ = Q.shape
    eye = np.broadcast_to(np.eye(b), (n, b, b))
    return np.linalg.solve(eye - Q, eye + Q)


def build_blocks(theta: np.ndarray, b: int, k: int) -> np.ndarray:
    """Packed parameters -> orthogonal (approximately) blocks [n][b][b]."""
    return cayley_neumann(unpack(theta, b), k)


# --------------------------------------------------------------------------
# Block-diagonal application  [tech-2-bd], input-centric order [tech-2-in]
# --------------------------------------------------------------------------

def apply_blockdiag(X: np.ndarray, blocks: np.ndarray) -> np.ndarray:
    """Row form of z_t = B x_t for block-diagonal B: token-major X [T][n*b],
    one independent product per block: out[:, g-block] = X[:, g-block] @ B_g^T."""
    X = np.asarray(X, dtype=np.float64)
    n, b, _ = blocks.shape
    out = np.empty((X.shape[0], n * b))
    for g in range(n):
        out[:, g * b:(g + 1) * b] = X[:, g * b:(g + 1) * b] @ blocks[g].T
    return out


def apply_blockdiag_transposed(X: np.ndarray, blocks: np.ndarray) -> np.ndarray:
    """Row form of z_t = B^T x_t: out[:, g-block] = X[:, g-block] @ B_g."""
    X = np.asarray(X, dtype=np.float64)
    n, b, _ = blocks.shape
    out = np.empty((X.shape[0], n * b))
    for g in range(n):
        out[:, g * b:(g + 1) * b] = X[:, g * b:(g + 1) * b] @ blocks[g]
    return out


def blockwise_outer(A: np.ndarray, B: np.ndarray, b: int) -> np.ndarray:
    """Per block g: sum_t A[t, g-block]^T (outer) B[t, g-block] -> [n][b][b]."""
    A = np.asarray(A, dtype=np.float64)
    B = np.asarray(B, dtype=np.float64)
    n = A.shape[1] // b
    G = np.empty((n, b, b))
    for g in range(n):
        G[g] = A[:, g * b:(g + 1) * b].T @ B[:, g * b:(g + 1) * b]
    return G


def forward(x, W0, P_blocks, R_blocks):
    """y_t = R_b (W0 (P_b x_t)) for every token.  Returns (y, u, v)."""
    x = np.asarray(x, dtype=np.float64)
    W0 = np.asarray(W0, dtype=np.float64)
    u = apply_blockdiag(x, P_blocks)        # u_t = P x_t
    v = u @ W0.T                            # v_t = W0 u_t
    y = apply_blockdiag(v, R_blocks)        # y_t = R v_t
    return y, u, v


def backward(dy, x, W0, P_blocks, R_blocks, v):
    """Gradients of L = sum_t <dy_t, y_t> with respect to x, P_b and R_b
    (W0 is frozen and gets none).  Returns (dx, G_P, G_R) where G_* are the
    gradients with respect to each full b x b block."""
    dy = np.asarray(dy, dtype=np.float64)
    x = np.asarray(x, dtype=np.float64)
    W0 = np.asarray(W0, dtype=np.float64)
    b = P_blocks.shape[1]
    dv = apply_blockdiag_transposed(dy, R_blocks)   # dv_t = R^T dy_t
    G_R = blockwise_outer(dy, v, b)                 # sum_t dy_t v_t^T
    du = dv @ W0                                    # du_t = W0^T dv_t
    G_P = blockwise_outer(du, x, b)                 # sum_t du_t x_t^T
    dx = apply_blockdiag_transposed(du, P_blocks)   # dx_t = P^T du_t
    return dx, G_P, G_R


def forward_v_rows(x, W0, P_blocks, rows):
    """v_t = W0 (P x_t) restricted to the output features `rows` (a slice):
    the same products as forward(), for a subset of its outputs."""
    u = apply_blockdiag(x, P_blocks)
    return u @ np.asarray(W0, dtype=np.float64)[rows].T


def backward_du_cols(dy, W0, R_blocks, cols):
    """du_t = W0^T (R^T dy_t) restricted to the input features `cols`."""
    dv = apply_blockdiag_transposed(dy, R_blocks)
    return dv @ np.asarray(W0, dtype=np.float64)[:, cols]


def cnp_adjoint(Q: np.ndarray, G: np.ndarray, k: int) -> np.ndarray:
    """Gradient with respect to Q of <G, R_k(Q)>, R_k = sum_i c_i Q^i.
    Written as the direct double sum of the derivative of each power:
        G_Q = sum_i c_i sum_{j=0}^{i-1} (Q^T)^j G (Q^T)^{i-1-j}."""
    c = neumann_coefficients(k)
    QT = np.transpose(Q, (0, 2, 1))
    pw = matrix_powers(QT, k)
    G_Q = np.zeros_like(G, dtype=np.float64)
    for i in range(1, k + 2):
        for j in range(i):
            G_Q += c[i] * (pw[j] @ G @ pw[i - 1 - j])
    return G_Q


def layer(theta_P, theta_R, W0, x, dy, b: int, k: int):
    """Whole hot path: build both sides, forward, backward, packed grads.
    Returns a dict of float64 arrays."""
    Q_P = unpack(theta_P, b)
    Q_R = unpack(theta_R, b)
    P_blocks = cayley_neumann(Q_P, k)
    R_blocks = cayley_neumann(Q_R, k)
    y, u, v = forward(x, W0, P_blocks, R_blocks)
    dx, G_P, G_R = backward(dy, x, W0, P_blocks, R_blocks, v)
    dtheta_P = pack_skew_grad(cnp_adjoint(Q_P, G_P, k))
    dtheta_R = pack_skew_grad(cnp_adjoint(Q_R, G_R, k))
    return dict(P_blocks=P_blocks, R_blocks=R_blocks, u=u, v=v, y=y, dx=dx,
                G_P=G_P, G_R=G_R, dtheta_P=dtheta_P, dtheta_R=dtheta_R)


def transform(theta, x, dout, b: int, k: int):
    """The block-diagonal transform on its own, z_t = B x_t, and the
    gradients of L = sum_t <dout_t, z_t> with respect to x and theta."""
    Q = unpack(theta, b)
    B = cayley_neumann(Q, k)
    z = apply_blockdiag(x, B)
    dx = apply_blockdiag_transposed(dout, B)
    G = blockwise_outer(dout, x, b)
    dtheta = pack_skew_grad(cnp_adjoint(Q, G, k))
    return dict(blocks=B, z=z, dx=dx, G=G, dtheta=dtheta)


# --------------------------------------------------------------------------
# Permuted blocks  [tech-2-perm], with explicit permutation matrices
# --------------------------------------------------------------------------

def permutation_matrix(perm) -> np.ndarray:
    """Pi with (Pi x)[i] = x[perm[i]]."""
    perm = np.asarray(perm)
    return np.eye(len(perm))[perm]


def layer_permuted(theta_P, theta_R, W0, x, dy, b: int, k: int, perm_P, perm_R):
    """The layer with permuted block-diagonal factors, written with dense
    matrices: R = Pi_R^T B_R Pi_R, P = Pi_P^T B_P Pi_P, y_t = R W0 P x_t.
    Gradients of L = sum_t <dy_t, y_t> by the chain rule through the dense
    matrices; the block gradients are the diagonal blocks of the dense
    gradients taken in the permuted basis."""
    x = np.asarray(x, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    W0 = np.asarray(W0, dtype=np.float64)
    Q_P = unpack(theta_P, b)
    Q_R = unpack(theta_R, b)
    BP = dense_from_blocks(cayley_neumann(Q_P, k))
    BR = dense_from_blocks(cayley_neumann(Q_R, k))
    PiP = permutation_matrix(perm_P)
    PiR = permutation_matrix(perm_R)
    P = PiP.T @ BP @ PiP
    R = PiR.T @ BR @ PiR
    y = x @ (R @ W0 @ P).T
    dx = dy @ (R @ W0 @ P)
    # dL/dBR = sum_t (Pi_R dy_t)(Pi_R W0 P x_t)^T ; dL/dBP = sum_t (Pi_P P^T... )
    a_R = dy @ PiR.T                      # rows: Pi_R dy_t
    c_R = x @ (PiR @ W0 @ P).T            # rows: Pi_R W0 P x_t
    dBR = a_R.T @ c_R
    a_P = dy @ (R @ W0 @ PiP.T)           # rows: Pi_P W0^T R^T dy_t
    c_P = x @ PiP.T                       # rows: Pi_P x_t
    dBP = a_P.T @ c_P
    nP, nR = BP.shape[0] // b, BR.shape[0] // b
    G_P = np.stack([dBP[g * b:(g + 1) * b, g * b:(g + 1) * b] for g in range(nP)])
    G_R = np.stack([dBR[g * b:(g + 1) * b, g * b:(g + 1) * b] for g in range(nR)])
    return dict(y=y, dx=dx,
                dtheta_P=pack_skew_grad(cnp_adjoint(Q_P, G_P, k)),
                dtheta_R=pack_skew_grad(cnp_adjoint(Q_R, G_R, k)))


def loss_permuted(theta_P, theta_R, W0, x, dy, b, k, perm_P, perm_R) -> float:
    BP = dense_from_blocks(build_blocks(theta_P, b, k))
    BR = dense_from_blocks(build_blocks(theta_R, b, k))
    PiP = permutation_matrix(perm_P)
    PiR = permutation_matrix(perm_R)
    W = PiR.T @ BR @ PiR @ np.asarray(W0, np.float64) @ PiP.T @ BP @ PiP
    y = np.asarray(x, np.float64) @ W.T
    return float(np.sum(np.asarray(dy, np.float64) * y))


# --------------------------------------------------------------------------
# Around the layer: merge and parameter update  [tech-2-merge]
# --------------------------------------------------------------------------

def merge(theta_P, theta_R, W0, b: int, k: int) -> np.ndarray:
    """W0 <- R W0 P with the current blocks, as dense matrices."""
    P = dense_from_blocks(build_blocks(theta_P, b, k))
    R = dense_from_blocks(build_blocks(theta_R, b, k))
    return R @ np.asarray(W0, dtype=np.float64) @ P


def adam_update(theta, grad, m, v, step: int, lr: float, beta1: float = 0.9,
                beta2: float = 0.999, eps: float = 1e-8, weight_decay: float = 0.0):
    """One Adam step on the packed parameters (Kingma and Ba, with bias
    correction; optional decoupled weight decay).  The pages do not name the
    optimizer of theta; this is the plain reading.  Returns (theta, m, v)."""
    theta = np.asarray(theta, dtype=np.float64)
    grad = np.asarray(grad, dtype=np.float64)
    m = beta1 * np.asarray(m, dtype=np.float64) + (1 - beta1) * grad
    v = beta2 * np.asarray(v, dtype=np.float64) + (1 - beta2) * grad * grad
    m_hat = m / (1 - beta1 ** step)
    v_hat = v / (1 - beta2 ** step)
    theta = theta - lr * (m_hat / (np.sqrt(v_hat) + eps) + weight_decay * theta)
    return theta, m, v


# --------------------------------------------------------------------------
# INT8 frozen weight  [tech-2-xq]
# --------------------------------------------------------------------------

def quantize_w0(W0):
    """Per-output-row symmetric INT8 codes and float32 scales of W0
    (float32 arithmetic: the division decides the integer code)."""
    W = np.asarray(W0, dtype=np.float32)
    d_out, d_in = W.shape
    codes = np.zeros((d_out, d_in), dtype=np.int8)
    scales = np.zeros(d_out, dtype=np.float32)
    for o in range(d_out):
        amax = np.float32(np.max(np.abs(W[o]))) if d_in else np.float32(0)
        s = np.float32(amax / np.float32(127))
        if s == 0:  # a zero row (or one whose scale underflows): codes 0
            continue
        scales[o] = s
        q = np.rint(W[o] / s)  # float32 quotient, ties to even
        codes[o] = np.clip(q, -127, 127).astype(np.int8)
    return codes, scales


def dequantize_w0(codes, scales):
    """W0[o][i] = code[o][i] * scale[o], one float32 product per entry."""
    q = np.asarray(codes, dtype=np.int8).astype(np.float32)
    s = np.asarray(scales, dtype=np.float32)
    return q * s[:, None]


# --------------------------------------------------------------------------
# Checks only: dense embedding and scalar loss for finite differences
# --------------------------------------------------------------------------

def dense_from_blocks(blocks: np.ndarray) -> np.ndarray:
    """Explicit d x d block-diagonal matrix (d = n*b)."""
    n, b, _ = blocks.shape
    D = np.zeros((n * b, n * b))
    for g in range(n):
        D[g * b:(g + 1) * b, g * b:(g + 1) * b] = blocks[g]
    return D


def loss(theta_P, theta_R, W0, x, dy, b: int, k: int) -> float:
    """L = sum_t <dy_t, y_t>, the scalar whose gradients backward() returns."""
    P_blocks = build_blocks(theta_P, b, k)
    R_blocks = build_blocks(theta_R, b, k)
    y, _, _ = forward(x, W0, P_blocks, R_blocks)
    return float(np.sum(np.asarray(dy, dtype=np.float64) * y))
