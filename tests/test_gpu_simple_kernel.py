"""The CUDA-core partial kernel (PD_PARTIAL_KERNEL=simple) stays an independent
cross-check of the tensor-core one: the small parity cases run against the
oracle in a child process with that kernel selected."""
import os
import subprocess
import sys

import pytest
import torch

from tests.conftest import ROOT

pytestmark = pytest.mark.gpu


def test_simple_partial_kernel_matches_oracle():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, PD_PARTIAL_KERNEL="simple")
    env.pop("PD_PARITY_LOG", None)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider", "-m",
                        "gpu", "tests/test_gpu_decode.py", "-k", "tiny or small_parity"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
