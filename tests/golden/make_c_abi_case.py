"""Writes c_abi_case_f32.bin: the inputs and the float64 oracle's outputs of
one small fp32 layer step, for the plain-C caller in tests/c_abi/.  Only the
seeded input generator and the oracle are used.

Layout (little-endian): 8 bytes "POETXC1\\0"; int32 d_in, d_out, b, k,
tokens; then float32 arrays in this order: theta_P [d_in/b][b(b-1)/2],
theta_R [d_out/b][b(b-1)/2], W0 [d_out][d_in], x [T][d_in], dy [T][d_out]
(inputs), y [T][d_out], dx [T][d_in], dtheta_P, dtheta_R (the oracle's
results rounded to float32).

Run from the repository root:  python tests/golden/make_c_abi_case.py
"""

import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from orthogonal_reparameterized_packed_gb300.inputs import make_layer_inputs  # noqa: E402

D_IN, D_OUT, B, K, T = 64, 32, 16, 2, 8


def main():
    inp = make_layer_inputs(D_IN, D_OUT, B, K, T, dtype="f32", sigma_theta=0.05, seed=42)
    ref = oracle.layer(inp.theta_P, inp.theta_R, inp.W0, inp.x, inp.dy, B, K)
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "c_abi_case_f32.bin")
    with open(out, "wb") as f:
        f.write(b"POETXC1\0")
        f.write(np.array([D_IN, D_OUT, B, K, T], dtype="<i4").tobytes())
        for a in (inp.theta_P, inp.theta_R, inp.W0, inp.x, inp.dy,
                  ref["y"], ref["dx"], ref["dtheta_P"], ref["dtheta_R"]):
            f.write(np.ascontiguousarray(a, dtype="<f4").tobytes())
    print(out)


if __name__ == "__main__":
    main()
