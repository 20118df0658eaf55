"""The bounds-checking build (libmsda_debug.so, MSDA_DEBUG_BOUNDS) on the GPU.

It runs in a child process that selects that library through MSDA_LIBRARY, so that the
rest of the suite keeps the normal build: every core, pruned, ordered and fused call in
tests/debug_bounds_cases.py must match the oracle and record no out-of-range corner row,
and the kernels' own check must report a made-up offender through
msda_debug_bounds_status.  Only in-range inputs are used: nothing here makes a kernel
access memory out of range.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_debug_build_checks_every_row_and_reports_an_offender():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a CUDA device")
    from scale_deformable_attention_msda3d_b300 import build
    lib = build.build(debug=True)
    env = dict(os.environ, MSDA_LIBRARY=lib)
    r = subprocess.run([sys.executable, os.path.join(HERE, "debug_bounds_cases.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, (r.stdout[-3000:], r.stderr[-3000:])
    assert "self-test reported" in r.stdout
