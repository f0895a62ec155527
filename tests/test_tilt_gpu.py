"""GPU parity of the tilted static split at the edges of its range.

CTAs of a launch start in blockIdx order as the previous grid's CTAs leave, so
the TMA kernels may give the late CTAs smaller static shares; the shares fall
with blockIdx down to zero rows at the extreme settings below. Whatever the
shares, every output row must be written once and match the oracle. The
library reads its scheduling variables once per process, so each setting runs
the cases of tilt_child.py in a child process.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))

SETTINGS = {
    "default": {},
    "linear, last share zero": {"PMG_SCHED_TILT_PCT": "100", "PMG_SCHED_TILT_POW": "1"},
    "quartic, last share zero": {"PMG_SCHED_TILT_PCT": "25", "PMG_SCHED_TILT_POW": "4"},
    "above the limit (clamped)": {"PMG_SCHED_TILT_PCT": "100", "PMG_SCHED_TILT_POW": "4"},
    "cubic, long head (per-token mode tilted too)": {"PMG_SCHED_TILT_PCT": "33", "PMG_SCHED_TILT_POW": "3",
                                                     "PMG_SCHED_HEAD_STAGES": "8"},
    "untilted": {"PMG_SCHED_TILT_PCT": "0"},
}


@pytest.mark.parametrize("setting", list(SETTINGS))
def test_tilted_split_matches_oracle(setting, cuda_lib):
    env = {k: v for k, v in os.environ.items() if not k.startswith("PMG_SCHED_")}
    env.update(SETTINGS[setting])
    r = subprocess.run([sys.executable, os.path.join(HERE, "tilt_child.py")], env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, f"child failed ({setting}):\n{r.stdout[-2000:]}\n{r.stderr[-4000:]}"
    assert "tilt-child ok 12" in r.stdout, r.stdout[-2000:]
