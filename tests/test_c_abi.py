"""The boundary is a C ABI: a plain C11 program (tests/c_abi_consumer.c)
compiled with gcc against include/afx.h and linked to libafx.so uses the
encoder, the header parser and the planner (host part, no GPU), and with
the CUDA runtime restores a container on the GPU and waits with afx_sync."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _compile(afx, tmp_path, gpu: bool):
    gcc = shutil.which("gcc")
    if not gcc:
        pytest.skip("gcc not available")
    lib_dir = os.path.dirname(afx.LIB_PATH)
    exe = str(tmp_path / ("consumer_gpu" if gpu else "consumer"))
    cmd = [gcc, "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c_abi_consumer.c"), "-o", exe, f"-L{lib_dir}", "-l:" + os.path.basename(afx.LIB_PATH),
           f"-Wl,-rpath,{lib_dir}"]
    if gpu:
        cuda = os.path.dirname(os.path.dirname(os.path.realpath(shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc")))
        cmd += ["-DAFX_CONSUMER_GPU", "-I", os.path.join(cuda, "include"), f"-L{os.path.join(cuda, 'lib64')}",
                "-lcudart", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe


def test_c_program_uses_the_host_abi(afx, tmp_path):
    exe = _compile(afx, tmp_path, gpu=False)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr


@pytest.mark.gpu
def test_c_program_restores_on_the_gpu(afx, tmp_path):
    exe = _compile(afx, tmp_path, gpu=True)
    r = subprocess.run([exe, "gpu"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
