"""include/gemm.h is a C header: a C99 program (tests/c_consumer.c) compiles
against it with -pedantic -Werror, links the library, and gets the plan of the
bf16 8192^3 + bias + GELU(tanh) product through host-only calls; the header also
compiles as C++."""
import os
import shutil
import subprocess

import pytest

import dense_gemm_bf16_gb300 as dg

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OUT = os.path.join(ROOT, "tests", "_build")


@pytest.fixture(scope="module")
def libdir():
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    dg.build()
    os.makedirs(OUT, exist_ok=True)
    return os.path.dirname(dg.library_path())


def test_c99_consumer_links_and_plans(libdir):
    exe = os.path.join(OUT, "c_consumer")
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                    "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_consumer.c"),
                    "-L", libdir, "-ldgemm_gb300", f"-Wl,-rpath,{libdir}", "-o", exe],
                   check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    first = r.stdout.splitlines()[0]
    assert first == ("kernel=1 block_m=128 block_n=256 block_k=128 stages=3 grid=152 "
                     "cta_pair=2 workspace=0")


def test_header_compiles_as_cpp():
    if shutil.which("g++") is None:
        pytest.skip("no C++ compiler")
    os.makedirs(OUT, exist_ok=True)
    src = os.path.join(OUT, "header_only.cpp")
    with open(src, "w") as f:
        f.write('#include "gemm.h"\nint main() { return gemm_set_option(GEMM_OPT_GROUP_M, 8) '
                '== GEMM_OK ? 0 : 1; }\n')
    subprocess.run(["g++", "-std=c++17", "-Wall", "-Wextra", "-Werror", "-pedantic", "-fsyntax-only",
                    "-I", os.path.join(ROOT, "include"), src],
                   check=True, capture_output=True, text=True)
