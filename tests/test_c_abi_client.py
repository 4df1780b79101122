"""The C ABI from plain C: tests/c/abi_client.c allocates its own device
buffers with the CUDA runtime, calls gdn_decode through include/lar.h and
checks the result against the fp64 oracle's C entry point.  Built with the
system C compiler; run on the GPU."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "abi_client.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _build_client(out_dir):
    import oracle
    from linear_attention_recurrent_gb300 import _build
    lar_lib = _build.LIB
    if not os.path.exists(lar_lib):
        pytest.skip("liblar.so is not built")
    ora_lib = oracle.build()
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = os.path.join(out_dir, "abi_client")
    rpath = ",".join(f"-rpath,{os.path.dirname(x)}" for x in (lar_lib, ora_lib))
    cmd = [cc, "-O2", "-std=c11", "-Wall", "-Werror", SRC, "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), "-o", exe, lar_lib, ora_lib,
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-lm", f"-Wl,{rpath}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_client_builds(tmp_path):
    """Compiles and links against liblar.so, the oracle and the CUDA runtime (no GPU needed)."""
    assert os.path.exists(_build_client(str(tmp_path)))


@pytest.mark.gpu
def test_c_client_matches_oracle(tmp_path, cuda_device):
    exe = _build_client(str(tmp_path))
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "gdn_decode_varlen match the oracle" in r.stdout
