"""The C ABI from plain C: tests/csrc/abi_consumer.c includes include/proj.h, is compiled
as strict C99 (warnings are errors) and linked against libhsp_proj.so.  On the CPU it
runs the queries and argument checks that need no device; on a GPU it allocates with the
CUDA runtime's C API, runs a fused and a separate call and checks every output exactly
(small integers) against its own double loop."""
import os
import shutil
import subprocess

import pytest

import hidden_state_projection_gb300 as hsp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "csrc", "abi_consumer.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _build(tmp_path, device: bool) -> str:
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(hsp.LIB_PATH)
    if not os.path.exists(hsp.LIB_PATH):
        pytest.skip("libhsp_proj.so is not built")
    exe = str(tmp_path / ("abi_consumer_dev" if device else "abi_consumer"))
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-O1",
           "-I", os.path.join(ROOT, "include"), SRC, "-o", exe,
           "-L", libdir, "-Wl,-rpath," + libdir, "-l:libhsp_proj.so"]
    if device:
        # the CUDA headers are not strict C99: system headers, exempt from -pedantic
        cmd[1:1] = ["-DABI_CONSUMER_DEVICE", "-isystem", os.path.join(CUDA, "include")]
        cudalib = os.path.join(CUDA, "lib64")
        cmd += ["-L", cudalib, "-Wl,-rpath," + cudalib, "-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_plain_c_build_and_host_checks(tmp_path):
    hsp.lib()
    exe = _build(tmp_path, device=False)
    r = subprocess.run([exe, "host"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr + r.stdout


@pytest.mark.gpu
def test_plain_c_device_calls_exact(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    hsp.lib()
    exe = _build(tmp_path, device=True)
    r = subprocess.run([exe, "device"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr + r.stdout


@pytest.mark.gpu
def test_plain_c_calls_survive_a_device_reset(tmp_path):
    """cudaDeviceReset in a child process (its own context only) between rounds of calls:
    the library's cached device addresses and kernel set-up follow the new context."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    hsp.lib()
    exe = _build(tmp_path, device=True)
    r = subprocess.run([exe, "reset"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr + r.stdout
