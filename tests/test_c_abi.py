"""The C ABI from C: tests/c/abi_stack.c includes only dlo.h and the CUDA
runtime header and drives a small DiT stack (layout, packing, registration,
forwards, statistics, slot checks, graphs, an argument error, teardown).  It
is compiled as strict C11 here (CPU) and run on the GPU."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "layerwise_weight_offload_slot_gb300")
SRC = os.path.join(ROOT, "tests", "c", "abi_stack.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _build(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    if not os.path.exists(os.path.join(PKG, "libdlo.so")):
        pytest.skip("libdlo.so is not built")
    if not os.path.exists(os.path.join(CUDA, "include", "cuda_runtime_api.h")):
        pytest.skip("no CUDA runtime headers")
    exe = str(tmp_path / "abi_stack")
    cmd = [cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-O2", SRC, "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), "-L", PKG, "-ldlo", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           "-lm", f"-Wl,-rpath,{PKG}", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_program_compiles_and_links_against_the_abi(tmp_path):
    assert os.path.exists(_build(tmp_path))


@pytest.mark.gpu
def test_c_program_drives_a_stack(tmp_path):
    exe = _build(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c abi ok" in r.stdout


def test_header_is_self_contained_in_c_and_cxx(tmp_path):
    """dlo.h compiles on its own (no CUDA or torch headers) as C99 and C++17."""
    src = tmp_path / "only_header.c"
    src.write_text('#include "dlo.h"\nint main(void) { dlo_desc d; (void)d; return DLO_OK; }\n')
    for compiler, flags in (("gcc", ["-std=c99", "-x", "c"]), ("g++", ["-std=c++17", "-x", "c++"])):
        cc = shutil.which(compiler)
        if cc is None:
            continue
        r = subprocess.run([cc, *flags, "-Wall", "-Wextra", "-Werror", "-fsyntax-only", "-I",
                            os.path.join(ROOT, "include"), str(src)], capture_output=True, text=True)
        assert r.returncode == 0, (compiler, r.stderr)
