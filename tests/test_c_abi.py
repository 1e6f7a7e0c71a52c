"""poetx.h is a C header: it compiles alone as ISO C99 (-pedantic), and a
plain C program (tests/c_abi/layer_step.c, C11 because the CUDA runtime's
own headers use anonymous unions) compiles against it with a C compiler, and on a GPU links against
libpoetx.so and runs one fp32 layer step (block build, forward, backward)
whose results are compared with stored float64-oracle values
(tests/golden/c_abi_case_f32.bin, written by make_c_abi_case.py from the
oracle only) at the fp32 tolerance, 1e-4 relative Frobenius."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi", "layer_step.c")
CASE = os.path.join(ROOT, "tests", "golden", "c_abi_case_f32.bin")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")
CFLAGS = ["-std=c11", "-pedantic", "-Wall", "-Wextra", "-Werror",
          "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include")]


def _cc():
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    return cc


def test_caller_compiles_as_c11():
    r = subprocess.run([_cc(), *CFLAGS, "-fsyntax-only", "-x", "c", SRC],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_header_alone_is_c99_clean(tmp_path):
    src = tmp_path / "h.c"
    src.write_text('#include "poetx.h"\nint main(void) { return (int)poetx_packed_size(4, 2); }\n')
    r = subprocess.run([_cc(), "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror",
                        "-fsyntax-only",
                        "-I", os.path.join(ROOT, "include"), str(src)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


@pytest.mark.gpu
def test_c_caller_layer_step_matches_stored_oracle(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import orthogonal_reparameterized_packed_gb300 as poetx
    lib = poetx.load_library()._name
    exe = tmp_path / "layer_step"
    libdir = os.path.dirname(lib)
    r = subprocess.run([_cc(), *CFLAGS, SRC, "-o", str(exe), "-L", libdir, "-lpoetx",
                        "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-lm",
                        f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe), CASE], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("OK"), r.stdout
