"""The FA_DEBUG build (libfa_debug.so): at the end of every pipelined kernel
(prefill, backward, GQA decode) the roles' protocol counts are compared, and a
mismatch is reported as FA_ERR_CHECK. A spread of calls through that build must
report nothing and give the regular build's outputs bit for bit: the checks
touch no arithmetic."""
import os
import subprocess
import sys

import numpy as np
import pytest

from parity import require_gpu

pytestmark = pytest.mark.gpu

TESTS = os.path.dirname(os.path.abspath(__file__))


def _run(lib, out):
    env = dict(os.environ, FA_LIBRARY=lib)
    r = subprocess.run([sys.executable, os.path.join(TESTS, "_debug_build_cases.py"), out], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert lib in r.stdout, r.stdout


def test_debug_build_checks_pass_and_change_nothing(tmp_path):
    require_gpu()
    from exact_attention_29_gb300 import build

    regular = build.build()
    debug = build.build(debug=True)
    _run(debug, str(tmp_path / "debug.npz"))
    _run(regular, str(tmp_path / "regular.npz"))
    a = np.load(tmp_path / "debug.npz")
    b = np.load(tmp_path / "regular.npz")
    assert sorted(a.files) == sorted(b.files) and len(a.files) > 30
    for name in a.files:
        assert np.array_equal(a[name], b[name], equal_nan=True), name
