"""The one-CTA-per-tile tensor-core kernels, which the library selects where a CTA pair does not
fit (B·L not a multiple of 256, d not a multiple of 256) and which DS_LOGITS_PAIR=0 /
DS_SELFCOND_PAIR=0 select always: the tensor-path step parity cases against the oracle, run in a
child process because the library reads those switches once per process."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("env", [{"DS_SELFCOND_PAIR": "0"},
                                 {"DS_SELFCOND_PAIR": "0", "DS_LOGITS_PAIR": "0"}],
                         ids=["selfcond_one_cta", "both_one_cta"])
def test_step_parity_with_one_cta_kernels(env):
    cmd = [sys.executable, "-m", "pytest", os.path.join("tests", "test_gpu_step.py"), "-q",
           "-p", "no:cacheprovider", "-m", "gpu", "-k",
           "(test_step_parity and tensor) or test_done_sequence_inside_a_pair_tile "
           "or test_race_beside_selfcond_matches_its_own_launch"]
    r = subprocess.run(cmd, cwd=ROOT, env={**os.environ, **env}, capture_output=True, text=True,
                       timeout=900)
    tail = (r.stdout + r.stderr)[-3000:]
    assert r.returncode == 0, tail
    assert " passed" in r.stdout and " failed" not in r.stdout, tail
