"""The debug-checks build of libyoco (built with YOCO_DEBUG_CHECKS): every kernel
checks the global indices it forms before using them and records a failed check
(never a trap).  On small valid cases of every call, its results must match the
oracle and no check may fail.  The release build says it has no checks."""
import ctypes
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


def _debug_lib():
    import importlib.util
    spec = importlib.util.spec_from_file_location("_yoco_build_dbg",
                                                  os.path.join(ROOT, "gated_retention_shared_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    if not os.path.exists(mod.DEBUG_LIB):
        mod.build(debug=True)
    return mod.DEBUG_LIB


def test_release_build_has_no_debug_checks():
    import gated_retention_shared_gb300 as Y
    w = ctypes.c_uint32(7)
    if os.environ.get("YOCO_LIB_PATH"):
        pytest.skip("this process runs another build")
    assert Y.lib.yoco_debug_checks(0, ctypes.byref(w)) == Y.YOCO_ERR_UNSUPPORTED


@pytest.mark.timeout(900)
def test_debug_build_small_cases_pass_every_check():
    lib = _debug_lib()
    env = dict(os.environ, YOCO_LIB_PATH=lib)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "_debug_cases.py")], env=env,
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "debug cases ok" in r.stdout
