"""The one-CTA-per-tile tensor-core kernels, which the library selects where a CTA pair does not
fit (B·L not a multiple of 256, d not a multiple of 256) and which DS_LOGITS_PAIR=0 /
DS_SELFCOND_PAIR=0 select always: the tensor-path step parity cases against the oracle, run in a
child process because the library reads those switches once per process."""
import os
import subprocess
import sys

import numpy as np
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


_CHILD = r"""
import sys
import numpy as np
import torch
sys.path.insert(0, "tests")
from _helpers import GpuCase, out_np
from canvas_sampler_gb300 import workloads as W
w = W.scaled(W.WORKLOADS["step_bf16_b8_v262144_d2816"], V=16384, d=512, B=2)
case = GpuCase(w)
outs = out_np(case.run_step(case.state()))
np.savez(sys.argv[1], **outs)
"""


def test_pair_and_one_cta_self_conditioning_agree_bit_for_bit(tmp_path):
    # the pair kernel issues the same MMAs in the same k order for every output element and
    # promotes the same TMEM chunks: s, the samples and the confidences must be identical
    res = {}
    for tag, env in (("pair", {}), ("one", {"DS_SELFCOND_PAIR": "0"})):
        path = tmp_path / f"{tag}.npz"
        r = subprocess.run([sys.executable, "-c", _CHILD, str(path)], cwd=ROOT,
                           env={**os.environ, **env}, capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, (r.stdout + r.stderr)[-3000:]
        res[tag] = dict(np.load(path))
    for k in res["pair"]:
        assert np.array_equal(res["pair"][k], res["one"][k]), k
