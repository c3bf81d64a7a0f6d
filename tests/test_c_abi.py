"""Plain C11 programs drive the library through include/pagedkv.h alone.

CPU: the programs compile as strict C11 against the header (the ABI is C,
not C++).  GPU: one runs a decode step and checks it against the C oracle;
the other runs a beam search (forks, copy on write) and checks every
beam's tokens and attention after each step.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "abi_step.c")
BEAM_SRC = os.path.join(ROOT, "tests", "c", "abi_beam.c")


def _cuda_home():
    nvcc = shutil.which("nvcc")
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc))) if nvcc else "/usr/local/cuda"


def _build(tmp_path, link, src=SRC):
    from oracle import build as ob
    from paged_kv_cache_162_gb300 import _build as lb
    cuda = _cuda_home()
    exe = str(tmp_path / os.path.splitext(os.path.basename(src))[0])
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-O1",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"), src]
    if not link:
        return subprocess.run(cmd + ["-c", "-o", exe + ".o"], capture_output=True, text=True)
    libs = [lb.build(), ob.build()]
    dirs = sorted({os.path.dirname(p) for p in libs} | {os.path.join(cuda, "lib64")})
    cmd += ["-o", exe] + [f"-L{d}" for d in dirs] + [f"-Wl,-rpath,{d}" for d in dirs]
    cmd += ["-l:libpagedkv.so", "-l:liboracle.so", "-lcudart", "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    return r if r.returncode else exe


@pytest.mark.parametrize("src", [SRC, BEAM_SRC], ids=["step", "beam"])
def test_header_and_caller_are_plain_c(tmp_path, src):
    r = _build(tmp_path, link=False, src=src)
    assert r.returncode == 0, r.stderr


@pytest.mark.gpu
def test_c_program_runs_a_step(tmp_path):
    exe = _build(tmp_path, link=True)
    assert isinstance(exe, str), getattr(exe, "stderr", exe)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c abi step ok" in r.stdout


@pytest.mark.gpu
def test_c_program_runs_a_beam_search(tmp_path):
    exe = _build(tmp_path, link=True, src=BEAM_SRC)
    assert isinstance(exe, str), getattr(exe, "stderr", exe)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c abi beam ok" in r.stdout
