"""The bounds-checked debug build (UPIPE_DEBUG_BOUNDS), the stand-in for a
memory checker: every plain (non-TMA) global load and store of the kernels is
checked against the extent of its view, and a failed check skips the access
and reports UPIPE_ERR_BOUNDS instead of touching memory."""
import ctypes
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _debug_lib():
    from headwise_chunked_attention_gb300.build import build
    return build(debug=True)


def test_debug_build_builds_and_exports_the_same_functions():
    # CPU: nvcc cross-compiles it; both builds declare which one they are
    from tests.test_host_abi import declared_functions
    from headwise_chunked_attention_gb300.build import build
    import headwise_chunked_attention_gb300 as u
    build()
    dbg = ctypes.CDLL(_debug_lib())
    rel = u.lib()
    for n in declared_functions():
        assert hasattr(dbg, n), n
    dbg.upipe_debug_bounds.restype = ctypes.c_int
    assert dbg.upipe_debug_bounds() == 1
    assert not u.DEBUG_BOUNDS and rel.upipe_debug_bounds() == 0
    dbg.upipe_strerror.restype = ctypes.c_char_p
    assert dbg.upipe_strerror(7) == b"device bounds check failed (debug build)"


@pytest.mark.gpu
def test_release_build_bounds_selftest_reports_nothing():
    # the release build compiles the checks away: the self-test's write (one
    # element past its declared view, inside its array) happens unreported
    import headwise_chunked_attention_gb300 as u
    assert u.selftest_bounds() is True
    assert u.last_error() == 0


@pytest.mark.gpu
def test_every_entry_point_passes_the_bounds_checks():
    # a child process (the binding picks its library once per process) runs
    # the forward, fused forward, both backwards with split query walks and
    # ragged and folding lengths on the debug build, against the oracle
    _debug_lib()
    env = dict(os.environ, UPIPE_DEBUG_BOUNDS="1", UPIPE_BWD_WALK="4")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "_debug_bounds_child.py")],
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "debug bounds ok" in r.stdout
