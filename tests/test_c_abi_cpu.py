"""include/fa.h is a C ABI: a plain C99 program compiles against it (gcc -std=c99 -pedantic, no
CUDA headers), links against libfa_gb300.so and gets the documented answers from the calls that
need no device."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not installed")
def test_c_program_uses_the_abi(lib_path, tmp_path):
    exe = tmp_path / "abi_from_c"
    src = os.path.join(ROOT, "tests", "c", "abi_from_c.c")
    libdir = os.path.dirname(lib_path)
    cc = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                         "-I", os.path.join(ROOT, "include"), src, "-L", libdir,
                         "-l:" + os.path.basename(lib_path), "-o", str(exe)],
                        capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr
    env = dict(os.environ, LD_LIBRARY_PATH=libdir + os.pathsep + os.environ.get("LD_LIBRARY_PATH", ""))
    run = subprocess.run([str(exe)], capture_output=True, text=True, env=env, timeout=120)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "abi 2." in run.stdout and "status0 ok" in run.stdout
