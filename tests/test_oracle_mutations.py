"""The pins catch plausible mistakes in the oracle.  Each case plants one
mistake in a copy of the oracle (a transposed operand, a flipped sign, a
dropped or extra term, a wrong index formula, a wrong rounding) in the layer,
its permuted variant, the merge, Adam and the INT8 weight, runs the pin tests
against the copy in a fresh interpreter and expects them to fail; the
unmodified copy must pass.  CPU only; the repository's oracle is never
touched."""

import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE = os.path.join(ROOT, "oracle", "poetx_oracle.py")

# (what the mistake is, text in the oracle, planted replacement)
MUTATIONS = [
    ("adjoint uses Q instead of Q^T", "QT = np.transpose(Q, (0, 2, 1))", "QT = Q"),
    ("forward block product not transposed",
     "out[:, g * b:(g + 1) * b] = X[:, g * b:(g + 1) * b] @ blocks[g].T",
     "out[:, g * b:(g + 1) * b] = X[:, g * b:(g + 1) * b] @ blocks[g]"),
    ("transposed block product transposed",
     "out[:, g * b:(g + 1) * b] = X[:, g * b:(g + 1) * b] @ blocks[g]\n",
     "out[:, g * b:(g + 1) * b] = X[:, g * b:(g + 1) * b] @ blocks[g].T\n"),
    ("skew projection with a plus", "G_Q[:, ii, jj] - G_Q[:, jj, ii]",
     "G_Q[:, ii, jj] + G_Q[:, jj, ii]"),
    ("Neumann coefficients: the top power dropped", "c[1: k + 2] += 1.0", "c[1: k + 1] += 1.0"),
    ("unpack without the minus sign", "Q[:, jj, ii] = -theta[:, idx]",
     "Q[:, jj, ii] = theta[:, idx]"),
    ("exact Cayley inverted", "return np.linalg.solve(eye - Q, eye + Q)",
     "return np.linalg.solve(eye + Q, eye - Q)"),
    ("dgrad with W0 transposed", "du = dv @ W0 ", "du = dv @ W0.T "),
    ("packed index off by a row", "return i * b - (i * (i + 1)) // 2 + (j - i - 1)",
     "return i * b - (i * (i - 1)) // 2 + (j - i - 1)"),
    ("token sum with its operands swapped",
     "G[g] = A[:, g * b:(g + 1) * b].T @ B[:, g * b:(g + 1) * b]",
     "G[g] = B[:, g * b:(g + 1) * b].T @ A[:, g * b:(g + 1) * b]"),
    ("power derivative with a wrong exponent", "G_Q += c[i] * (pw[j] @ G @ pw[i - 1 - j])",
     "G_Q += c[i] * (pw[j] @ G @ pw[i - j])"),
    ("permuted factor conjugated the wrong way", "P = PiP.T @ BP @ PiP", "P = PiP @ BP @ PiP.T"),
    ("permuted block gradient transposed", "dBP = a_P.T @ c_P", "dBP = c_P.T @ a_P"),
    ("merge with R transposed", "return R @ np.asarray(W0, dtype=np.float64) @ P",
     "return R.T @ np.asarray(W0, dtype=np.float64) @ P"),
    ("Adam without the first moment's bias correction", "m_hat = m / (1 - beta1 ** step)",
     "m_hat = m"),
    ("Adam second moment of the raw gradient", "(1 - beta2) * grad * grad", "(1 - beta2) * grad"),
    ("Adam weight decay with the wrong sign", "+ weight_decay * theta)", "- weight_decay * theta)"),
    ("INT8 scale over 128 steps", "s = np.float32(amax / np.float32(127))",
     "s = np.float32(amax / np.float32(128))"),
    ("INT8 codes truncated instead of rounded", "q = np.rint(W[o] / s)", "q = np.floor(W[o] / s)"),
    ("dequantisation divides by the scale", "return q * s[:, None]", "return q / s[:, None]"),
    ("sampled v: W0's columns instead of its rows",
     "return u @ np.asarray(W0, dtype=np.float64)[rows].T",
     "return u @ np.asarray(W0, dtype=np.float64)[:, rows].T"),
    ("sampled v: W0 not transposed", "return u @ np.asarray(W0, dtype=np.float64)[rows].T",
     "return u @ np.asarray(W0, dtype=np.float64).T[rows]"),
    ("sampled du: W0's rows instead of its columns",
     "return dv @ np.asarray(W0, dtype=np.float64)[:, cols]",
     "return dv @ np.asarray(W0, dtype=np.float64)[cols].T"),
    ("sampled du: R applied untransposed",
     "dv = apply_blockdiag_transposed(dy, R_blocks)\n    return dv @ np.asarray(W0",
     "dv = apply_blockdiag(dy, R_blocks)\n    return dv @ np.asarray(W0"),
]


@pytest.fixture(scope="module")
def tree(tmp_path_factory):
    """A copy of what the pin tests import: the oracle, the input generator
    package (Python files only), the pins and their golden files."""
    dst = tmp_path_factory.mktemp("mut")
    shutil.copytree(os.path.join(ROOT, "oracle"), dst / "oracle",
                    ignore=shutil.ignore_patterns("__pycache__"))
    pkg = "orthogonal_reparameterized_packed_gb300"
    os.makedirs(dst / pkg)
    for f in os.listdir(os.path.join(ROOT, pkg)):
        if f.endswith(".py"):
            shutil.copy(os.path.join(ROOT, pkg, f), dst / pkg / f)
    os.makedirs(dst / "tests")
    for f in ("conftest.py", "test_oracle_pins.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), dst / "tests" / f)
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), dst / "tests" / "golden")
    return dst


def run_pins(tree):
    env = dict(os.environ, PYTHONDONTWRITEBYTECODE="1")
    return subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                           str(tree / "tests" / "test_oracle_pins.py")],
                          cwd=str(tree), capture_output=True, text=True, env=env, timeout=600)


def test_unmodified_copy_passes(tree):
    r = run_pins(tree)
    assert r.returncode == 0, r.stdout[-3000:]


@pytest.mark.parametrize("what,text,planted", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_fails_a_pin(tree, what, text, planted):
    src = open(ORACLE).read()
    assert src.count(text) == 1, f"anchor for '{what}' not found once in the oracle"
    target = tree / "oracle" / "poetx_oracle.py"
    try:
        target.write_text(src.replace(text, planted, 1))
        r = run_pins(tree)
    finally:
        target.write_text(src)
    assert r.returncode != 0, f"no pin caught: {what}"
