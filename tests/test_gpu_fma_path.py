"""The fp32-FMA instantiation of the attention kernel (the comparison the
tensor-core path is measured against) meets the same parity bar.  It runs in a
child process because the path is chosen once per process (GK_ATTN_PATH)."""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu


def test_fma_path_parity():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    here = os.path.dirname(os.path.abspath(__file__))
    env = dict(os.environ, GK_ATTN_PATH="fma")
    r = subprocess.run([sys.executable, os.path.join(here, "gk_fma_check.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    assert "fma path ok" in r.stdout
