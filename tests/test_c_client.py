"""The C ABI from plain C: tests/c/kvq_c_client.c (C99, the CUDA runtime's C
API and include/kvq.h only) compiled with gcc against libkvq.so.  On the host
the program must compile and link (the header is valid C, every symbol it
calls is exported); on the GPU it runs its exact-by-construction cases."""
import os
import shutil
import subprocess

import pytest

import kv_quant_cache_gb300 as kvq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "kvq_c_client.c")
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _compile(out_dir):
    gcc = shutil.which("gcc")
    if gcc is None or not os.path.exists(os.path.join(CUDA_HOME, "include", "cuda_runtime.h")):
        pytest.skip("gcc or the CUDA runtime headers are not available")
    kvq.lib()  # the library is built
    pkg = os.path.dirname(kvq.LIB_PATH)
    exe = os.path.join(out_dir, "kvq_c_client")
    cmd = [gcc, "-std=c99", "-O2", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA_HOME, "include"),
           SRC, "-o", exe, "-L", pkg, "-lkvq", "-L", os.path.join(CUDA_HOME, "lib64"), "-lcudart",
           f"-Wl,-rpath,{pkg}", f"-Wl,-rpath,{os.path.join(CUDA_HOME, 'lib64')}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


def test_c_client_compiles_and_links(tmp_path):
    assert os.path.exists(_compile(str(tmp_path)))


def test_header_is_valid_cpp(tmp_path):
    """include/kvq.h also compiles as C++ (extern "C" linkage, no C-only
    constructs)."""
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not available")
    src = tmp_path / "use_header.cpp"
    src.write_text('#include "kvq.h"\nint main() { return kvq_status_string(KVQ_OK) ? 0 : 1; }\n')
    r = subprocess.run([gxx, "-std=c++17", "-Wall", "-Wextra", "-Werror", "-fsyntax-only",
                        "-I", os.path.join(ROOT, "include"), str(src)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr


@pytest.mark.gpu
def test_c_client_runs(tmp_path, cuda_device):
    exe = _compile(str(tmp_path))
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c client ok" in r.stdout
