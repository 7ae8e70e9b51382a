"""A C program calls the library through include/gemm.h alone.

`-m "not gpu"`: the header compiles as C (gcc -std=c11 -Wall -Werror) and the
program links against libgemm.so.  `-m gpu`: the program runs and checks its
results against its own double-precision loop.
"""
import os
import subprocess

import pytest

from stage_software_pipelining_gb300 import build as gemm_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_consumer", "main.c")


def compile_consumer(tmp_path):
    lib = gemm_build.build()
    exe = os.path.join(tmp_path, "gemm_c_consumer")
    libdir = os.path.dirname(lib)
    subprocess.run(["gcc", "-std=c11", "-O2", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    SRC, "-o", exe, "-L", libdir, "-lgemm", f"-Wl,-rpath,{libdir}", "-lm"],
                   check=True, capture_output=True, text=True)
    return exe


def test_header_compiles_as_c_and_links(tmp_path):
    assert os.path.exists(compile_consumer(tmp_path))


@pytest.mark.gpu
def test_c_program_runs_on_the_gpu(tmp_path, gpu):
    exe = compile_consumer(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "0 entries out of tolerance" in r.stdout
