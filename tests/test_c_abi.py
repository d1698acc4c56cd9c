"""The C ABI from C: include/ptoc.h compiles as C99 and as C++ (CPU), and a
plain C program that owns its buffers (cudaMalloc) drives the library and
checks closed-form results (GPU); a plain C program runs the host credit
barrier with POSIX threads as ranks (CPU)."""
import os
import shutil
import subprocess

import pytest

from conftest import ROOT

import tile_level_collective_gb300 as P

CUDA = "/usr/local/cuda"


def cuda_include():
    for d in (os.path.join(CUDA, "include"), os.path.join(CUDA, "targets", "sbsa-linux", "include"),
              os.path.join(CUDA, "targets", "x86_64-linux", "include")):
        if os.path.exists(os.path.join(d, "cuda_runtime_api.h")):
            return d
    pytest.skip("CUDA headers not found")


@pytest.mark.parametrize("lang,std,cc", [("c", "c99", "gcc"), ("c", "c11", "gcc"), ("c++", "c++17", "g++")])
def test_header_compiles(lang, std, cc, tmp_path):
    src = tmp_path / "h.c"
    src.write_text('#include "ptoc.h"\nint f(void) { return (int)PTOC_MAX_RANKS + (int)PTOC_ATOMIC_ADD; }\n')
    r = subprocess.run([cc, "-x", lang, "-std=" + std, "-Wall", "-Wextra", "-Werror", "-fsyntax-only",
                        "-I", os.path.join(ROOT, "include"), "-I", cuda_include(), str(src)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


@pytest.mark.gpu
def test_plain_c_caller(tmp_path):
    exe = tmp_path / "abi_check"
    libdir = os.path.dirname(P.LIB_PATH)
    cudalib = [d for d in (os.path.join(CUDA, "lib64"), os.path.join(CUDA, "lib"))
               if os.path.exists(d)]
    cmd = ["gcc", "-std=c11", "-O1", "-o", str(exe), os.path.join(ROOT, "tests", "c", "abi_check.c"),
           "-I", os.path.join(ROOT, "include"), "-I", cuda_include(), "-L", libdir, "-lptoc",
           "-Wl,-rpath," + libdir]
    for d in cudalib:
        cmd += ["-L", d, "-Wl,-rpath," + d]
    cmd += ["-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "abi_check: ok" in r.stdout


def test_plain_c_host_barrier(tmp_path):
    """ptoc_credit_barrier_host from C with POSIX threads as ranks (no GPU):
    complete calls self-clear, an absent rank leaves the protocol's credits."""
    exe = tmp_path / "host_barrier_check"
    libdir = os.path.dirname(P.LIB_PATH)
    cmd = ["gcc", "-std=c11", "-O1", "-pthread", "-o", str(exe),
           os.path.join(ROOT, "tests", "c", "host_barrier_check.c"),
           "-I", os.path.join(ROOT, "include"), "-I", cuda_include(), "-L", libdir, "-lptoc",
           "-Wl,-rpath," + libdir]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "host barrier: ok" in r.stdout
