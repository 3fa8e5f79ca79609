"""GPU: the sm_103 reducing TMEM load that the varlen softmax uses for the row
max of tiles that need no mask (tcgen05.ld.red ... .max, the helper
tmem_ld32_max) returns the stored values unchanged and a maximum bitwise equal
to the software maximum of the same values, -inf included.  The probe in
tests/probes is compiled with nvcc against the library's own PTX helpers and
run as its own process."""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(REPO, "varlen_flashattention_forward_gb300", "csrc")
PROBE = os.path.join(REPO, "tests", "probes", "tmem_ld_red_max.cu")


def test_tmem_ld_red_max_equals_software_max(cuda_device, tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = str(tmp_path / "tmem_ld_red_max")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-I", CSRC, "-o", exe, PROBE], check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "PASS" in r.stdout, r.stdout
