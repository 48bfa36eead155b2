"""The range-checked debug library (build(debug=True), loaded with
FM_LIBRARY=debug): its kernels check every shared-memory address, TMA
coordinate and TMEM lane / column before handing it to the hardware. Every
attention kernel (d = 64, 128, 256; bf16 and FP8 forwards; both backwards) runs
clean under it at parity with the oracle."""
import os
import subprocess
import sys

import pytest

from mask_aware_sparse_gb300 import build as fmbuild

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_debug_build_runs_every_kernel_clean():
    fmbuild.build(debug=True)
    env = dict(os.environ, FM_LIBRARY="debug")
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_build_case.py")], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "debug build clean" in r.stdout
