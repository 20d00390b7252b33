"""The C ABI driven from a plain C program (tests/c_abi/abi_smoke.c): no Python
binding and no torch on the path.  The program allocates with the CUDA runtime,
calls arx_reduce (separate and in-place output, every W, ragged n),
arx_step in each barrier variant, arx_step_noalloc, arx_reduce_host on
page-locked buffers and the external-writer form (arx_ext_post as the producer,
arx_ext_step as the consumer), and compares every output bit for bit with the
CPU oracle's C library.  Compiled with gcc on the machine that runs it."""

import os
import shutil
import subprocess

import pytest

from conftest import ROOT

pytestmark = pytest.mark.gpu

CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def test_c_program_against_the_oracle(product_lib_path, tmp_path):
    import oracle.build
    oracle_lib = oracle.build.build()
    cc = shutil.which(os.environ.get("CC", "gcc"))
    assert cc, "a C compiler is needed to build the C ABI test"
    exe = str(tmp_path / "abi_smoke")
    lib_dir = os.path.dirname(product_lib_path)
    orc_dir = os.path.dirname(oracle_lib)
    cmd = [cc, "-O2", "-std=c11", "-Wall", "-Wextra",
           os.path.join(ROOT, "tests", "c_abi", "abi_smoke.c"), "-o", exe,
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           "-L", lib_dir, "-l:libarx.so", "-L", orc_dir, "-l:liboracle.so",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           f"-Wl,-rpath,{lib_dir}:{orc_dir}:{os.path.join(CUDA, 'lib64')}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, f"compile failed:\n{r.stderr}"
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "c abi ok" in r.stdout, f"rc={r.returncode}\n{r.stdout}\n{r.stderr}"
