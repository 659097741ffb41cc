"""The DSPARK_CHECKED build: every gather site checks its index, records a violation in the
status word and never traps.

The test compiles that build into a temporary directory, runs the cases of tests/_checked_cases.py
through it in a child process (DSPARK_LIBRARY names the checked library) and through the default
build here, and compares: clean cases leave no status bit and give identical outputs in both
builds; each planted out-of-range caller index is flagged through dspark_read_status as
INPUT_RANGE by both builds and additionally as INDEX by the checked one, with the same
substituted outputs.
"""
import json
import os
import subprocess
import sys

import pytest

from tests._checked_cases import run_cases

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PLANTED = ("markov_anchor", "markov_tc_anchor", "reduced_table", "verify_token", "confidence_token")


def test_checked_build_flags_planted_indices_without_faulting(cuda_lib, tmp_path):
    from draft_sampling_verification_tcgen05_gb300 import _build
    lib = _build.build(force=True, extra_flags=["-DDSPARK_CHECKED"], lib_path=str(tmp_path / "libdspark_checked.so"),
                       build_dir=str(tmp_path / "obj"))
    result = tmp_path / "checked.json"
    env = dict(os.environ, DSPARK_LIBRARY=lib)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "_checked_cases.py"), str(result), ROOT],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    checked = json.loads(result.read_text())
    assert checked.pop("_library") == lib
    plain = run_cases(cuda_lib)
    assert set(plain) == set(checked)
    for name in plain:
        pb, cb = plain[name].pop("bits"), checked[name].pop("bits")
        assert plain[name] == checked[name], f"{name}: outputs differ between the builds"
        assert not pb & cuda_lib.STATUS_INDEX, f"{name}: the default build set INDEX"
        if name in PLANTED:
            assert pb & cuda_lib.STATUS_INPUT_RANGE, f"{name}: default build did not flag the planted index"
            assert cb & cuda_lib.STATUS_INPUT_RANGE and cb & cuda_lib.STATUS_INDEX, \
                f"{name}: checked build bits {cb:#x}"
        else:
            assert pb == 0 and cb == 0, f"{name}: clean case flagged ({pb:#x}, {cb:#x})"
    # the planted index changed only what it touches
    assert plain["reduced_table"]["tokens"][0][1] == -1
    assert all(t == -1 for t in plain["verify_token"]["tokens"][2])
