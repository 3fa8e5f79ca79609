"""GPU: the gather ceiling of the sparse-MLA decode structure.

The probe in tests/probes copies the decode workload's gathered rows (2048
rows of 1152 bytes per token, random positions on 64-row pages of a 4.8 GB
paged cache) through the decode kernel's two-stage chunked ring with the same
cp.async gather, but does no attention: its rate is the most the decode
kernel's gather can deliver at a given CTA count (one CTA per token).  The
test checks that every wait finished (no TIMEOUT), that the rates are
plausible for HBM3e, and prints them; the bench reports the decode kernel's
own rate next to the measured copy peak.
"""
import os
import re
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(REPO, "varlen_flashattention_forward_gb300", "csrc")
PROBE = os.path.join(REPO, "tests", "probes", "gather_ceiling.cu")


def test_gather_ceiling(cuda_device, tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = str(tmp_path / "gather_ceiling")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-I", CSRC, "-o", exe, PROBE], check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    print(r.stdout)
    assert r.returncode == 0, r.stdout + r.stderr
    rates = {}
    for m in re.finditer(r"gather ctas=(\d+) threads=(\d+): ([\d.]+) us (\d+) GB/s", r.stdout):
        rates[(int(m.group(1)), int(m.group(2)))] = float(m.group(4))
    assert (128, 128) in rates and len(rates) >= 2, r.stdout
    for gbs in rates.values():
        assert 500.0 < gbs < 9000.0, r.stdout
