"""The prefill kernels kept for comparison (PKV_PREFILL_KERNEL=tc1: the
tcgen05 kernel with one query tile per CTA, which also serves the cascade's
prefix pass; =mma: the mma.sync kernel), each checked against the oracle in a
child process (GPU)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("kernel", ["tc1", "mma"])
def test_prefill_comparison_kernel(kernel, cuda_device):
    env = dict(os.environ, PKV_PREFILL_KERNEL=kernel)
    env["PYTHONPATH"] = os.pathsep.join([HERE, os.path.dirname(HERE), env.get("PYTHONPATH", "")])
    r = subprocess.run([sys.executable, os.path.join(HERE, "prefill_case_check.py")], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    assert "ok" in r.stdout
