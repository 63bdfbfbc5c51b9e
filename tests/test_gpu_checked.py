"""The checked build (DFLASH_CHECKED=1: device-side index checks that record DF_ERR_BOUNDS
instead of touching memory) runs the acceptance and mixture-of-experts parity tests green:
every check holds on valid inputs, and the results match the oracle as in the default build."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_checked_build_passes_accept_and_moe_parity():
    env = dict(os.environ, DFLASH_CHECKED="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-p", "no:cacheprovider",
                        "tests/test_gpu_accept.py", "tests/test_gpu_moe.py"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert os.path.exists(os.path.join(ROOT, "block_diffusion_draft_dflash_gb300", "_build_checked", "libdflash.so"))
