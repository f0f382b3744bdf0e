"""The bounds-checked build (-DADAMW_CHECK_BOUNDS=1, the stand-in for a
memory sanitizer): every kernel checks each chunk against its tensor's
buffers before touching it.  Builds that variant into a temporary folder
and runs tests/bounds_check_run.py against it in a child process: every
storage mode over ragged and long lists (also lists whose last rounds are
claimed at run time), clipped (fused and not) and device-resident steps,
must run with no chunk refused and bit-identical to the oracle; a chunk
lengthened past its tensor must be refused, reported in the device status
word and left unwritten."""
import os
import subprocess
import sys

import pytest

from adamw_optimizer_step_sm_gb300 import build as B

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_bounds_checked_build_refuses_nothing_valid_and_catches_a_bad_chunk(tmp_path):
    lib = B.build(defines=["ADAMW_CHECK_BOUNDS=1"], out_dir=str(tmp_path / "chk"))
    env = dict(os.environ, ADAMW_SM_LIBRARY=lib,
               PYTHONPATH=os.pathsep.join([HERE, B.ROOT, os.environ.get("PYTHONPATH", "")]))
    r = subprocess.run([sys.executable, os.path.join(HERE, "bounds_check_run.py")], env=env,
                       capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "a lengthened chunk was refused" in r.stdout


def test_default_build_does_not_check_and_refuses_to_lengthen_chunks():
    import torch
    from adamw_optimizer_step_sm_gb300 import adamw_sm as A
    assert A.adamw_build_flags() & A.BUILD_CHECK_BOUNDS == 0
    t = [torch.zeros(4096, dtype=torch.bfloat16, device="cuda") for _ in range(5)]
    plan = A.Plan([t[0]], [t[1]], [t[2]], [t[3]], [t[4]], A.MODE_BF16_KAHAN)
    with pytest.raises(A.AdamWError) as e:
        A.adamw_plan_test_corrupt_chunk(plan.handle, 0, 8)
    assert e.value.status == A.ADAMW_ERR_INVALID_ARG
    plan.close()
