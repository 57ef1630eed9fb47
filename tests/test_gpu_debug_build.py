"""The bounds-checked debug build (nvcc -DVT_CHECKS, libvt_gb300_checks.so).

Every kernel of that build tests the indices of its index-computed global
accesses, skips an access that would leave its buffer and records the
source line.  Here: the reporting path works (a kernel whose check fails by
design, inside an in-bounds buffer), and every GPU test (parity, canaries,
error words) passes under the checked build with no failed check (conftest
asserts that after every GPU test when VT_CHECKS=1)."""
import os
import subprocess
import sys

import pytest
import torch

import frequency_ranked_drafter_gb300 as vt
from gpu_util import need_cuda

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SENTINEL = 0xFFFFFFFF


def test_check_selftest_reports_in_either_build():
    """Release build: all n + 1 values written, nothing reported.  Checked
    build: the last write skipped and its check's line reported once."""
    dev = need_cuda()
    lib = vt.load()
    n = 1000
    buf = torch.full((n + 1,), -1, dtype=torch.int32, device=dev)
    rc = lib.vt_selftest_check(buf.data_ptr(), n,
                               torch.cuda.current_stream().cuda_stream)
    assert rc == 0, lib.vt_last_error()
    torch.cuda.synchronize()
    got = buf.cpu()
    assert torch.equal(got[:n], torch.arange(n, dtype=torch.int32))
    if lib.vt_debug_build():
        assert int(got[n]) == -1
        assert lib.vt_debug_checks() > 0
        assert lib.vt_debug_checks() == 0  # read and cleared
    else:
        assert int(got[n]) == n
        assert lib.vt_debug_checks() == 0


def test_suites_pass_under_the_checked_build():
    need_cuda()
    if os.environ.get("VT_CHECKS", "") == "1":
        pytest.skip("already running under the checked build")
    env = dict(os.environ, VT_CHECKS="1")
    r = subprocess.run(
        [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu",
         "-p", "no:cacheprovider", os.path.join(ROOT, "tests")],
        env=env, cwd=ROOT, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
