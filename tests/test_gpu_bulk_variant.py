"""The optional cp.async.bulk staging of the bf16 Kahan update
(-DADAMW_BULK=1, measured slower than the default and not used by it):
builds that variant into a temporary folder and runs
tests/bulk_variant_run.py against it in a child process, which checks its
bf16 Kahan paths against the oracle bit for bit."""
import os
import subprocess
import sys

import pytest

from adamw_optimizer_step_sm_gb300 import build as B

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_staging_build_matches_the_oracle(tmp_path):
    lib = B.build(defines=["ADAMW_BULK=1"], out_dir=str(tmp_path / "bulk"))
    env = dict(os.environ, ADAMW_SM_LIBRARY=lib,
               PYTHONPATH=os.pathsep.join([HERE, B.ROOT, os.environ.get("PYTHONPATH", "")]))
    r = subprocess.run([sys.executable, os.path.join(HERE, "bulk_variant_run.py")], env=env,
                       capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "bit-identical to the oracle" in r.stdout
