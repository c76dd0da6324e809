"""The bounds-checked debug build, libep_gb300_checked.so (loaded with EP_GB300_CHECKED=1).

That build checks every index that comes from data against the buffer it indexes; a failure
skips the access and sets EP_STATUS_BOUNDS in the layout's status word instead of faulting.
1. The parity suites run unchanged against it in a child process.  On valid inputs no check
   may fire (every status comparison with the oracle would fail on a stray EP_STATUS_BOUNDS),
   and every output must still equal the oracle's.
2. A layout a caller has overwritten with rows outside [0, R_max) goes through every entry
   point in both builds.  Both skip those rows (guard rows past R_max stay untouched); only the
   checked build reports them, as EP_STATUS_BOUNDS and EP_ERR_BOUNDS."""
import json
import os
import subprocess
import sys

import pytest

import __graft_entry__ as entry

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.join(ROOT, "tests")


def _checked_env():
    entry._load_builder().build(checked=True)
    env = dict(os.environ)
    env["EP_GB300_CHECKED"] = "1"
    env["PYTHONPATH"] = os.pathsep.join([ROOT, TESTS, env.get("PYTHONPATH", "")])
    return env


def test_parity_suites_pass_on_the_checked_build():
    suites = ["test_gpu_parity.py", "test_gpu_padded.py", "test_gpu_fuzz.py", "test_gpu_fp8.py",
              "test_gpu_edge.py", "test_gpu_routing_map.py"]
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           "-k", "not largest_token_count"] + [os.path.join(TESTS, s) for s in suites]
    r = subprocess.run(cmd, cwd=ROOT, env=_checked_env(), capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    assert " passed" in r.stdout


def test_corrupted_rows_are_skipped_and_reported():
    import combine_topk_ids_histogram_gb300 as ep
    from checked_cases import run_corrupted_rows

    got = run_corrupted_rows(ep)                         # the default build, in this process
    assert not got["checked"]
    assert got["guards_untouched"] and got["outputs_finite"]
    assert got["status"] == 0 and got["read_status_rc"] == ep.EP_OK

    code = ("import json, checked_cases, combine_topk_ids_histogram_gb300 as ep; "
            "assert ep.CHECKED and ep.LIB_PATH.endswith('libep_gb300_checked.so'); "
            "print(json.dumps(checked_cases.run_corrupted_rows(ep)))")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=_checked_env(), capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    chk = json.loads(r.stdout.strip().splitlines()[-1])
    assert chk["checked"] and chk["lib"].endswith("libep_gb300_checked.so")
    assert chk["guards_untouched"] and chk["outputs_finite"]
    assert chk["status"] & ep.STATUS_BOUNDS
    assert chk["read_status_rc"] == ep.EP_ERR_BOUNDS
