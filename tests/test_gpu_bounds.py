"""The bounds-checked build (libdlr_checked.so: every guarded shared- and global-memory index
checked on the device, a violation skipping the access and reported through the status word),
which stands in for a memory checker. Its cases run in a child process with
DLR_BOUNDS_CHECK=1 (the binding loads one library per process): every entry point on small,
ragged shapes, each result within the oracle's tolerance, no check failing; and the self-test
whose one planted out-of-range read the check skips and reports."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def result():
    env = dict(os.environ, DLR_BOUNDS_CHECK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "bounds_cases.py")],
                       env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stderr[-4000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_the_checked_library_ran(result):
    assert result["checked"] is True
    assert result["library"].endswith("libdlr_checked.so")
    assert len(result["cases"]) >= 30


def test_no_index_check_fails_and_results_match_the_oracle(result):
    for name, err, status, site in result["cases"]:
        assert status == 0, f"{name}: device status {status} (site {site})"
        assert site == 0, f"{name}: bounds check failed at site {site}"
        tol = 1e-2 if "bf16" in name else 1e-5
        assert err <= tol, f"{name}: rel L2 {err:.3e}"


def test_planted_out_of_range_read_is_caught(result):
    status, site = result["selftest"]
    assert status == 6  # DLR_ERR_BOUNDS
    assert site // 100000 == 14 and site % 100000 > 0  # the self-test kernel's file and line
