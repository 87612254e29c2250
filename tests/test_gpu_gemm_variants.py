"""Run the grouped-GEMM parity tests once per kernel variant.  The kernel
choice is read from MOE_GEMM_2SM once per process, so each variant runs in a
child process: 0 = 1-SM kernel (128x256 tiles), 256 = CTA-pair kernel with
256x256 tiles, 128 = CTA-pair kernel with 256x128 tiles."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("variant", ["0", "256", "128"])
def test_gemm_parity_per_kernel_variant(variant):
    env = dict(os.environ, MOE_GEMM_2SM=variant)
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(HERE, "test_gpu_gemm.py"), "-m", "gpu", "-q",
                        "-p", "no:cacheprovider"], env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]


def test_nvfp4_parity_on_the_pair_kernel():
    """NVFP4 FWD/DGRAD run on the 1-SM kernel by default; MOE_GEMM_2SM=256
    selects the CTA-pair kernel's NVFP4 instance, which must pass the same
    parity tests."""
    env = dict(os.environ, MOE_GEMM_2SM="256")
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(HERE, "test_gpu_nvfp4.py"), "-m", "gpu", "-q",
                        "-p", "no:cacheprovider", "-k", "grouped_gemm"], env=env, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
