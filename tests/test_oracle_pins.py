"""Pins for the float64 oracle: each test checks it against something other
than itself (brute-force enumeration, closed forms, invariants of the
mathematics, an independent dense construction, finite differences), so
that a dropped term, a wrong sign or index or a transposed operand in the
oracle fails at least one of them.  CPU only."""

import json
import os

import numpy as np
import pytest
import scipy.linalg

import oracle
from orthogonal_reparameterized_packed_gb300.inputs import make_layer_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_skew(rng, n, b, scale):
    M = rng.standard_normal((n, b, b)) * scale
    return M - np.transpose(M, (0, 2, 1))


# ----------------------------------------------------------------- packing

@pytest.mark.parametrize("b", [2, 3, 5, 8, 32, 64])
def test_packed_index_matches_enumeration(b):
    count = 0
    for i in range(b):
        for j in range(i + 1, b):
            assert oracle.packed_index(i, j, b) == count
            count += 1
    assert count == oracle.packed_size(b)


@pytest.mark.parametrize("b", [2, 4, 7, 32])
def test_unpack_is_inverse_of_enumerated_pack(b):
    rng = np.random.default_rng(1)
    A = _rand_skew(rng, 3, b, 1.0)
    theta = np.zeros((3, oracle.packed_size(b)))
    for g in range(3):
        c = 0
        for i in range(b):
            for j in range(i + 1, b):
                theta[g, c] = A[g, i, j]
                c += 1
    Q = oracle.unpack(theta, b)
    assert np.array_equal(Q, A)
    assert np.array_equal(Q, -np.transpose(Q, (0, 2, 1)))
    assert np.all(np.diagonal(Q, axis1=1, axis2=2) == 0)


@pytest.mark.parametrize("b", [2, 5, 16])
def test_pack_skew_grad_matches_enumeration(b):
    rng = np.random.default_rng(2)
    G = rng.standard_normal((2, b, b))
    got = oracle.pack_skew_grad(G)
    for g in range(2):
        c = 0
        for i in range(b):
            for j in range(i + 1, b):
                assert got[g, c] == G[g, i, j] - G[g, j, i]
                c += 1


def test_neumann_coefficients():
    assert list(oracle.neumann_coefficients(0)) == [1, 1]
    assert list(oracle.neumann_coefficients(3)) == [1, 2, 2, 2, 1]


# ----------------------------------------------------- 2x2 closed forms

def _two_by_two(a):
    return oracle.unpack(np.array([[a]]), 2)


def test_golden_2x2_rotation():
    """Closed-form 2x2 values stored in tests/golden (see its header)."""
    with open(os.path.join(GOLDEN, "cayley_2x2.json")) as f:
        gold = json.load(f)
    for case in gold["cases"]:
        Q = _two_by_two(case["a"])
        np.testing.assert_allclose(oracle.cayley_exact(Q)[0], case["cayley"],
                                   rtol=0, atol=1e-15)
        for k_str, R in case["neumann"].items():
            np.testing.assert_allclose(oracle.cayley_neumann(Q, int(k_str))[0], R,
                                       rtol=0, atol=1e-15)


@pytest.mark.parametrize("a", [0.0, 0.1, -0.37, 0.9])
@pytest.mark.parametrize("k", [0, 1, 2, 3, 4, 5])
def test_2x2_neumann_closed_form(a, k):
    # Q = [[0,a],[-a,0]] has Q^2 = -a^2 I, so sum_{i<=k} Q^i = alpha I + beta Q
    alpha = sum((-a * a) ** m for m in range(k // 2 + 1))
    beta = sum((-a * a) ** m for m in range((k - 1) // 2 + 1)) if k >= 1 else 0.0
    diag = alpha - beta * a * a
    off = alpha + beta
    want = np.array([[diag, off * a], [-off * a, diag]])
    got = oracle.cayley_neumann(_two_by_two(a), k)[0]
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-15)


# ------------------------------------------------------- exact Cayley

@pytest.mark.parametrize("b,scale", [(8, 0.3), (32, 0.1), (64, 0.05), (16, 2.0)])
def test_exact_cayley_is_orthogonal(b, scale):
    rng = np.random.default_rng(3)
    Q = _rand_skew(rng, 4, b, scale)
    C = oracle.cayley_exact(Q)
    for g in range(4):
        err = np.max(np.abs(C[g].T @ C[g] - np.eye(b)))
        assert err <= 1e-12
        assert abs(np.linalg.det(C[g]) - 1.0) < 1e-10


@pytest.mark.parametrize("k", [0, 1, 2, 3, 5, 8])
def test_neumann_truncation_error_closed_form(k):
    # C - R_k = (I+Q) Q^{k+1} (I-Q)^{-1}; Q is normal with eigenvalues i*lam,
    # |1+i lam| = |1-i lam|, so ||C - R_k||_2 = ||Q||_2^{k+1} exactly.
    rng = np.random.default_rng(4)
    b = 24
    Q = _rand_skew(rng, 3, b, 0.08)
    C = oracle.cayley_exact(Q)
    R = oracle.cayley_neumann(Q, k)
    I = np.eye(b)
    for g in range(3):
        rhs = (I + Q[g]) @ np.linalg.matrix_power(Q[g], k + 1) @ np.linalg.inv(I - Q[g])
        np.testing.assert_allclose(C[g] - R[g], rhs, rtol=0, atol=1e-12)
        rho = np.linalg.norm(Q[g], 2)
        err = np.linalg.norm(C[g] - R[g], 2)
        assert abs(err - rho ** (k + 1)) <= 1e-9 * max(1.0, rho ** (k + 1))


def test_neumann_error_shrinks_with_k():
    rng = np.random.default_rng(5)
    Q = _rand_skew(rng, 2, 32, 0.05)
    C = oracle.cayley_exact(Q)
    errs = [np.linalg.norm(C - oracle.cayley_neumann(Q, k)) for k in range(7)]
    rho = max(np.linalg.norm(Q[g], 2) for g in range(2))
    assert rho < 1
    for k in range(1, 7):
        assert errs[k] < errs[k - 1]
        assert errs[k] / errs[k - 1] <= rho * 1.0001


# ---------------------------------------- forward: dense and spectrum

def _dense_reference(theta_P, theta_R, W0, b, k):
    """Independent dense construction with scipy's block_diag."""
    P = scipy.linalg.block_diag(*oracle.build_blocks(theta_P, b, k))
    R = scipy.linalg.block_diag(*oracle.build_blocks(theta_R, b, k))
    return R @ np.asarray(W0, np.float64) @ P


@pytest.mark.parametrize("d_in,d_out,b", [(16, 24, 4), (32, 32, 8), (12, 12, 12)])
def test_blockdiag_path_equals_dense_product(d_in, d_out, b):
    inp = make_layer_inputs(d_in, d_out, b, 3, 7, dtype="f32", sigma_theta=0.2, seed=6)
    W = _dense_reference(inp.theta_P, inp.theta_R, inp.W0, b, 3)
    P = oracle.build_blocks(inp.theta_P, b, 3)
    R = oracle.build_blocks(inp.theta_R, b, 3)
    y, _, _ = oracle.forward(inp.x, inp.W0, P, R)
    want = np.asarray(inp.x, np.float64) @ W.T
    np.testing.assert_allclose(y, want, rtol=0, atol=1e-13 * np.abs(want).max())


def test_spectrum_preserved_with_exact_cayley():
    rng = np.random.default_rng(7)
    d_in, d_out, b = 32, 24, 8
    W0 = rng.standard_normal((d_out, d_in))
    CP = oracle.cayley_exact(_rand_skew(rng, d_in // b, b, 0.4))
    CR = oracle.cayley_exact(_rand_skew(rng, d_out // b, b, 0.4))
    # W from the input-centric forward: feeding x = I gives y = W^T
    y, _, _ = oracle.forward(np.eye(d_in), W0, CP, CR)
    W = y.T
    s0 = np.linalg.svd(W0, compute_uv=False)
    s = np.linalg.svd(W, compute_uv=False)
    np.testing.assert_allclose(s, s0, rtol=1e-10, atol=0)
    # the truncated series is not exactly orthogonal: its spectrum moves
    PK = oracle.cayley_neumann(_rand_skew(np.random.default_rng(8), d_in // b, b, 0.4), 1)
    yk, _, _ = oracle.forward(np.eye(d_in), W0, PK, CR)
    sk = np.linalg.svd(yk.T, compute_uv=False)
    assert np.max(np.abs(sk - s0) / s0) > 1e-4


# ------------------------------------------------------ special cases

def test_zero_theta_gives_identity_blocks_and_plain_linear():
    inp = make_layer_inputs(16, 8, 4, 3, 5, dtype="f32", seed=9)
    zP = np.zeros_like(inp.theta_P)
    zR = np.zeros_like(inp.theta_R)
    out = oracle.layer(zP, zR, inp.W0, inp.x, inp.dy, 4, 3)
    assert np.array_equal(out["P_blocks"], np.broadcast_to(np.eye(4), (4, 4, 4)))
    x = inp.x.astype(np.float64)
    W0 = inp.W0.astype(np.float64)
    dy = inp.dy.astype(np.float64)
    np.testing.assert_allclose(out["y"], x @ W0.T, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(out["dx"], dy @ W0, rtol=1e-14, atol=1e-14)
    # R_k'(0)[H] = 2H: dtheta_R = pack(2(G_R - G_R^T)) with G_R = sum_t dy_t v_t^T
    v = x @ W0.T
    G_R = np.einsum("tgi,tgj->gij", dy.reshape(5, 2, 4), v.reshape(5, 2, 4))
    want = np.zeros_like(out["dtheta_R"])
    c = 0
    for i in range(4):
        for j in range(i + 1, 4):
            want[:, c] = 2 * (G_R[:, i, j] - G_R[:, j, i])
            c += 1
    np.testing.assert_allclose(out["dtheta_R"], want, rtol=1e-13, atol=1e-13)


def test_k0_is_one_plus_q():
    rng = np.random.default_rng(10)
    Q = _rand_skew(rng, 3, 6, 0.3)
    np.testing.assert_array_equal(oracle.cayley_neumann(Q, 0), np.eye(6) + Q)


def test_single_block_b_equals_d():
    inp = make_layer_inputs(8, 8, 8, 2, 3, dtype="f32", sigma_theta=0.3, seed=11)
    P = oracle.build_blocks(inp.theta_P, 8, 2)[0]
    R = oracle.build_blocks(inp.theta_R, 8, 2)[0]
    y, _, _ = oracle.forward(inp.x, inp.W0, P[None], R[None])
    want = inp.x.astype(np.float64) @ (R @ inp.W0.astype(np.float64) @ P).T
    np.testing.assert_allclose(y, want, rtol=1e-13, atol=1e-13)


# ------------------------------------- sliced products (sampled checks)

@pytest.mark.parametrize("rows", [slice(0, 24), slice(4, 8), slice(13, 22)])
def test_forward_v_rows_equals_dense_w0_p(rows):
    # d_out != d_in, so a slip between W0's rows and columns cannot pass
    inp = make_layer_inputs(16, 24, 4, 3, 7, dtype="f32", sigma_theta=0.2, seed=30)
    P = oracle.build_blocks(inp.theta_P, 4, 3)
    W = np.asarray(inp.W0, np.float64) @ scipy.linalg.block_diag(*P)  # W0 P, dense
    want = np.asarray(inp.x, np.float64) @ W.T
    got = oracle.forward_v_rows(inp.x, inp.W0, P, rows)
    assert got.shape == want[:, rows].shape
    np.testing.assert_allclose(got, want[:, rows], rtol=0, atol=1e-13 * np.abs(want).max())


@pytest.mark.parametrize("cols", [slice(0, 16), slice(4, 8), slice(9, 14)])
def test_backward_du_cols_equals_dense_rt_w0(cols):
    inp = make_layer_inputs(16, 24, 4, 3, 7, dtype="f32", sigma_theta=0.2, seed=31)
    R = oracle.build_blocks(inp.theta_R, 4, 3)
    # du_t = W0^T R^T dy_t, i.e. rows du = dy R W0 with dense R
    want = np.asarray(inp.dy, np.float64) @ scipy.linalg.block_diag(*R) @ \
        np.asarray(inp.W0, np.float64)
    got = oracle.backward_du_cols(inp.dy, inp.W0, R, cols)
    assert got.shape == want[:, cols].shape
    np.testing.assert_allclose(got, want[:, cols], rtol=0, atol=1e-13 * np.abs(want).max())


def test_sliced_products_give_the_sampled_block_gradients():
    # the block gradients built from the sliced products equal the full
    # backward's (FD-pinned) G_R and G_P block by block
    inp = make_layer_inputs(8, 12, 4, 3, 6, dtype="f32", sigma_theta=0.3, seed=32)
    P = oracle.build_blocks(inp.theta_P, 4, 3)
    R = oracle.build_blocks(inp.theta_R, 4, 3)
    _, _, v = oracle.forward(inp.x, inp.W0, P, R)
    _, G_P, G_R = oracle.backward(inp.dy, inp.x, inp.W0, P, R, v)
    for g in range(3):
        sl = slice(4 * g, 4 * g + 4)
        G = oracle.blockwise_outer(inp.dy[:, sl], oracle.forward_v_rows(inp.x, inp.W0, P, sl), 4)
        np.testing.assert_allclose(G[0], G_R[g], rtol=1e-12, atol=1e-13)
    for g in range(2):
        sl = slice(4 * g, 4 * g + 4)
        du = oracle.backward_du_cols(inp.dy, inp.W0, R, sl)
        G = oracle.blockwise_outer(du, inp.x[:, sl], 4)
        np.testing.assert_allclose(G[0], G_P[g], rtol=1e-12, atol=1e-13)


# ------------------------------------------------- finite differences

def _central_diff(f, x0, idx, h):
    xp = x0.copy()
    xm = x0.copy()
    xp[idx] += h
    xm[idx] -= h
    return (f(xp) - f(xm)) / (2 * h)


@pytest.mark.parametrize("k", [0, 1, 3])
def test_gradients_match_central_differences(k):
    inp = make_layer_inputs(8, 12, 4, k, 5, dtype="f32", sigma_theta=0.3, seed=12)
    tP = inp.theta_P.astype(np.float64)
    tR = inp.theta_R.astype(np.float64)
    x = inp.x.astype(np.float64)
    W0 = inp.W0.astype(np.float64)
    dy = inp.dy.astype(np.float64)
    out = oracle.layer(tP, tR, W0, x, dy, 4, k)
    h = 1e-6

    def rel(a, b):
        return abs(a - b) / max(1e-8, abs(b))

    for idx in np.ndindex(*tP.shape):
        fd = _central_diff(lambda t: oracle.loss(t, tR, W0, x, dy, 4, k), tP, idx, h)
        assert rel(out["dtheta_P"][idx], fd) <= 1e-6
    for idx in np.ndindex(*tR.shape):
        fd = _central_diff(lambda t: oracle.loss(tP, t, W0, x, dy, 4, k), tR, idx, h)
        assert rel(out["dtheta_R"][idx], fd) <= 1e-6
    for idx in [(0, 0), (2, 5), (4, 7), (1, 3)]:
        fd = _central_diff(lambda xx: oracle.loss(tP, tR, W0, xx, dy, 4, k), x, idx, h)
        assert rel(out["dx"][idx], fd) <= 1e-6


def test_cnp_adjoint_matches_directional_derivative():
    # unconstrained direction H (not skew) checks the full adjoint
    rng = np.random.default_rng(13)
    b, k = 6, 4
    Q = _rand_skew(rng, 1, b, 0.3)
    G = rng.standard_normal((1, b, b))
    H = rng.standard_normal((1, b, b))
    G_Q = oracle.cnp_adjoint(Q, G, k)
    eps = 1e-6
    f = lambda t: np.sum(G * oracle.cayley_neumann(Q + t * H, k))
    fd = (f(eps) - f(-eps)) / (2 * eps)
    assert abs(np.sum(G_Q * H) - fd) <= 1e-7 * max(1.0, abs(fd))


def test_transform_gradients_match_central_differences():
    inp = make_layer_inputs(12, 12, 4, 3, 6, dtype="f32", sigma_theta=0.3, seed=14)
    th = inp.theta_P.astype(np.float64)
    x = inp.x.astype(np.float64)
    g = inp.dy.astype(np.float64)
    out = oracle.transform(th, x, g, 4, 3)

    def L(t, xx):
        return float(np.sum(g * oracle.apply_blockdiag(xx, oracle.build_blocks(t, 4, 3))))

    for idx in np.ndindex(*th.shape):
        fd = _central_diff(lambda t: L(t, x), th, idx, 1e-6)
        assert abs(out["dtheta"][idx] - fd) <= 1e-6 * max(1e-8, abs(fd))
    for idx in [(0, 0), (3, 11), (5, 6)]:
        fd = _central_diff(lambda xx: L(th, xx), x, idx, 1e-6)
        assert abs(out["dx"][idx] - fd) <= 1e-6 * max(1e-8, abs(fd))
    # block-diagonal application against scipy's dense block_diag
    D = scipy.linalg.block_diag(*out["blocks"])
    np.testing.assert_allclose(out["z"], x @ D.T, rtol=0, atol=1e-13)


# ------------------------------------------------- permuted blocks

def test_permuted_layer_with_identity_permutations_is_the_plain_layer():
    inp = make_layer_inputs(12, 8, 4, 3, 5, dtype="f32", sigma_theta=0.3, seed=15)
    a = oracle.layer(inp.theta_P, inp.theta_R, inp.W0, inp.x, inp.dy, 4, 3)
    p = oracle.layer_permuted(inp.theta_P, inp.theta_R, inp.W0, inp.x, inp.dy, 4, 3,
                              np.arange(12), np.arange(8))
    for name in ("y", "dx", "dtheta_P", "dtheta_R"):
        np.testing.assert_allclose(p[name], a[name], rtol=1e-12, atol=1e-12)


def test_permutation_matrix_gathers():
    perm = np.array([2, 0, 3, 1])
    x = np.array([10.0, 11.0, 12.0, 13.0])
    assert list(oracle.permutation_matrix(perm) @ x) == [12.0, 10.0, 13.0, 11.0]


def test_permuted_layer_gradients_match_central_differences():
    rng = np.random.default_rng(16)
    inp = make_layer_inputs(8, 12, 4, 2, 4, dtype="f32", sigma_theta=0.3, seed=17)
    pP, pR = rng.permutation(8), rng.permutation(12)
    tP = inp.theta_P.astype(np.float64)
    tR = inp.theta_R.astype(np.float64)
    x = inp.x.astype(np.float64)
    W0 = inp.W0.astype(np.float64)
    dy = inp.dy.astype(np.float64)
    out = oracle.layer_permuted(tP, tR, W0, x, dy, 4, 2, pP, pR)

    def L(a, c, xx):
        return oracle.loss_permuted(a, c, W0, xx, dy, 4, 2, pP, pR)

    for idx in np.ndindex(*tP.shape):
        fd = _central_diff(lambda t: L(t, tR, x), tP, idx, 1e-6)
        assert abs(out["dtheta_P"][idx] - fd) <= 1e-6 * max(1e-8, abs(fd))
    for idx in np.ndindex(*tR.shape):
        fd = _central_diff(lambda t: L(tP, t, x), tR, idx, 1e-6)
        assert abs(out["dtheta_R"][idx] - fd) <= 1e-6 * max(1e-8, abs(fd))
    for idx in [(0, 1), (3, 7)]:
        fd = _central_diff(lambda xx: L(tP, tR, xx), x, idx, 1e-6)
        assert abs(out["dx"][idx] - fd) <= 1e-6 * max(1e-8, abs(fd))
    # y from the dense product
    assert np.allclose(out["y"], x @ (oracle.permutation_matrix(pR).T
                                      @ oracle.dense_from_blocks(oracle.build_blocks(tR, 4, 2))
                                      @ oracle.permutation_matrix(pR) @ W0
                                      @ oracle.permutation_matrix(pP).T
                                      @ oracle.dense_from_blocks(oracle.build_blocks(tP, 4, 2))
                                      @ oracle.permutation_matrix(pP)).T)


# ------------------------------------------------- merge and update

def test_merge_equals_the_layer_with_zero_theta():
    # after W0' = R W0 P, the layer with theta = 0 (identity blocks) gives the
    # same y as the layer with theta on the old W0
    inp = make_layer_inputs(16, 12, 4, 3, 6, dtype="f32", sigma_theta=0.3, seed=18)
    W1 = oracle.merge(inp.theta_P, inp.theta_R, inp.W0, 4, 3)
    a = oracle.layer(inp.theta_P, inp.theta_R, inp.W0, inp.x, inp.dy, 4, 3)
    z = oracle.layer(np.zeros_like(inp.theta_P), np.zeros_like(inp.theta_R), W1, inp.x, inp.dy,
                     4, 3)
    np.testing.assert_allclose(z["y"], a["y"], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(z["dx"], a["dx"], rtol=1e-12, atol=1e-12)
    # zero parameters leave W0 unchanged
    W2 = oracle.merge(np.zeros_like(inp.theta_P), np.zeros_like(inp.theta_R), inp.W0, 4, 3)
    assert np.array_equal(W2, inp.W0.astype(np.float64))


def test_adam_first_step_closed_form():
    # m = v = 0 at step 1: m_hat = g, v_hat = g^2, update = lr g / (|g| + eps)
    g = np.array([0.5, -2.0, 1e-3, 0.0])
    th, m, v = oracle.adam_update(np.zeros(4), g, np.zeros(4), np.zeros(4), 1, lr=0.1, eps=1e-8)
    np.testing.assert_allclose(th, -0.1 * g / (np.abs(g) + 1e-8), rtol=1e-12, atol=0)
    np.testing.assert_allclose(m, 0.1 * g)
    np.testing.assert_allclose(v, 0.001 * g * g)


def test_adam_second_step_by_hand():
    g1, g2 = 0.3, -0.7
    th, m, v = oracle.adam_update(np.array([1.0]), np.array([g1]), np.zeros(1), np.zeros(1), 1,
                                  lr=0.01, weight_decay=0.1)
    th, m, v = oracle.adam_update(th, np.array([g2]), m, v, 2, lr=0.01, weight_decay=0.1)
    m_want = 0.9 * 0.1 * g1 + 0.1 * g2
    v_want = 0.999 * 0.001 * g1 * g1 + 0.001 * g2 * g2
    th1 = 1.0 - 0.01 * (g1 / (abs(g1) + 1e-8) + 0.1 * 1.0)
    th2 = th1 - 0.01 * ((m_want / (1 - 0.81)) / (np.sqrt(v_want / (1 - 0.999 ** 2)) + 1e-8)
                        + 0.1 * th1)
    np.testing.assert_allclose(th, [th2], rtol=1e-12)
    np.testing.assert_allclose(m, [m_want], rtol=1e-12)
    np.testing.assert_allclose(v, [v_want], rtol=1e-12)


# ------------------------------------------------------- INT8 frozen weight

def test_quantize_rows_with_exact_scales():
    # amax 127 gives scale 1 and amax 63.5 gives scale 0.5 exactly, so the
    # codes are the round-half-even of the entries (or of twice them).
    W = np.array([[127.0, 3.25, -64.5, 2.5, 0.0],
                  [63.5, 1.25, -0.75, 0.5, -63.5]], dtype=np.float32)
    q, s = oracle.quantize_w0(W)
    assert s.dtype == np.float32 and q.dtype == np.int8
    assert s.tolist() == [1.0, 0.5]
    assert q.tolist() == [[127, 3, -64, 2, 0], [127, 2, -2, 1, -127]]
    assert np.array_equal(oracle.dequantize_w0(q, s),
                          np.array([[127, 3, -64, 2, 0], [63.5, 1, -1, 0.5, -63.5]],
                                   dtype=np.float32))


def test_quantize_zero_row_and_nearest_code():
    rng = np.random.default_rng(50)
    W = (rng.standard_normal((6, 200)) / np.sqrt(200)).astype(np.float32)
    W[3] = 0
    q, s = oracle.quantize_w0(W)
    assert s[3] == 0 and not q[3].any()
    assert np.all(oracle.dequantize_w0(q, s)[3] == 0)
    for o in (0, 1, 2, 4, 5):
        # the row's largest entry takes the largest code; every code is the
        # nearest integer to W / scale (checked against the neighbours)
        assert np.max(np.abs(q[o].astype(int))) == 127
        assert int(q[o][np.argmax(np.abs(W[o]))]) == int(np.sign(W[o][np.argmax(np.abs(W[o]))])) * 127
        ratio = W[o].astype(np.float64) / np.float64(s[o])
        err = np.abs(ratio - q[o])
        assert np.all(err <= 0.5 + 1e-5)
        assert np.all(err <= np.abs(ratio - (q[o] + 1)) + 1e-9)
        assert np.all(err <= np.abs(ratio - (q[o] - 1)) + 1e-9)
        # the round trip is within half a step
        deq = oracle.dequantize_w0(q[o:o + 1], s[o:o + 1])[0].astype(np.float64)
        assert np.all(np.abs(deq - W[o]) <= 0.5 * s[o] * (1 + 1e-5))


def test_quantize_scale_and_sign_symmetry():
    rng = np.random.default_rng(51)
    W = rng.standard_normal((4, 64)).astype(np.float32)
    q, s = oracle.quantize_w0(W)
    qn, sn = oracle.quantize_w0(-W)
    assert np.array_equal(sn, s) and np.array_equal(qn, -q)
    # a power-of-two scaling of a row scales its scale and keeps its codes
    q2, s2 = oracle.quantize_w0(W * np.float32(4))
    assert np.array_equal(q2, q) and np.array_equal(s2, s * 4)
