"""The bounds-checked build of the same sources (libswin_attn_bounds.so,
compiled with -DSWIN_CHECK_BOUNDS): every global load and store that a
kernel addresses itself (land bytes, LSE values, output rows, dBias partial
tables, the fp32 path's token rows) is range-checked against its buffer
first; a violation would be recorded in the plan's status word and the
access skipped. Every parity test asserts a clean status word, so running
them against that build shows that no kernel addressed outside its buffers
on those cases. They run in a child process, which loads the checked build
instead of the product library."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_parity_cases_on_the_bounds_checked_build():
    from shifted_window_attention_cyclic_gb300 import build
    build.build(check_bounds=True)
    env = dict(os.environ, SWIN_ATTN_CHECK_BOUNDS="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "gpu", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_gpu_parity.py"),
                        "-k", "small_sweep or tables_bit_exact or (full_parity and ragged) or all_land"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, (r.stdout[-3000:], r.stderr[-2000:])
    assert " passed" in r.stdout
